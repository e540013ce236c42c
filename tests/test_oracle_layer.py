"""Pins of the oracle's layer math: pure-Python loops (math module only) on tiny
inputs, textbook special cases and invariants.

Layer structure: QKV projections, attention, output projection and an MLP whose
weights are four h x h and two h x h2 matrices (FlexGen paper explainer, "Cost Model
and Policy Search", the 8*h1^2 + 4*h1*h2 weight term); pre-LN and ReLU come from the
workload definition; readings R5-R10 are stated in ``oracle/layer.py``.
"""
import math

import numpy as np
import pytest

import fg_synth
from oracle import layer as OL
from oracle import quant as Q


# ----------------------------------------------------------------------------- loops


def ln_loop(row, g, b, eps):
    n = len(row)
    mu = sum(row) / n
    var = sum((v - mu) ** 2 for v in row) / n
    return [(v - mu) / math.sqrt(var + eps) * gg + bb for v, gg, bb in zip(row, g, b)]


def matvec_loop(x, W, bias):
    K, N = len(W), len(W[0])
    return [sum(x[k] * W[k][n] for k in range(K)) + bias[n] for n in range(N)]


def attn_loop(q, ks, vs, d):
    """softmax over positions of q.k/sqrt(d), applied to v (one head)."""
    sc = [sum(qi * ki for qi, ki in zip(q, k)) / math.sqrt(d) for k in ks]
    m = max(sc)
    e = [math.exp(s - m) for s in sc]
    z = sum(e)
    return [sum(e[t] * vs[t][j] for t in range(len(ks))) / z for j in range(len(vs[0]))]


def tolist(a):
    return np.asarray(a, dtype=np.float64).tolist()


# ----------------------------------------------------------------------------- tests


def test_layernorm_loop_and_moments():
    r = np.random.Generator(np.random.PCG64(11))
    x = r.standard_normal((3, 96)) * 3 + 1
    g = r.standard_normal(96)
    b = r.standard_normal(96)
    y = OL.layernorm(x, g, b, 1e-5)
    for i in range(3):
        assert np.allclose(y[i], ln_loop(tolist(x[i]), tolist(g), tolist(b), 1e-5),
                           rtol=0, atol=1e-12)
    y1 = OL.layernorm(x, np.ones(96), np.zeros(96), 0.0)
    assert np.allclose(y1.mean(-1), 0, atol=1e-12)
    assert np.allclose(y1.var(-1), 1, atol=1e-12)


def test_causal_attention_loop():
    r = np.random.Generator(np.random.PCG64(12))
    S, T, H, d = 2, 5, 2, 4
    q, k, v = (r.standard_normal((S, T, H * d)) for _ in range(3))
    o = OL.causal_attention(q, k, v, H, d)
    for s in range(S):
        for i in range(T):
            for hh in range(H):
                sl = slice(hh * d, hh * d + d)
                ref = attn_loop(tolist(q[s, i, sl]), [tolist(k[s, j, sl]) for j in range(i + 1)],
                                [tolist(v[s, j, sl]) for j in range(i + 1)], d)
                assert np.allclose(o[s, i, sl], ref, rtol=0, atol=1e-12)


def test_attention_special_cases():
    r = np.random.Generator(np.random.PCG64(13))
    T, H, d = 6, 2, 8
    v = r.standard_normal((1, T, H * d))
    k = r.standard_normal((1, T, H * d))
    # position 0 sees only itself: output = v_0
    o = OL.causal_attention(r.standard_normal((1, T, H * d)), k, v, H, d)
    assert np.allclose(o[0, 0], v[0, 0], atol=1e-14)
    # equal scores (q = 0): position i outputs the mean of v_0..v_i
    o = OL.causal_attention(np.zeros((1, T, H * d)), k, v, H, d)
    for i in range(T):
        assert np.allclose(o[0, i], v[0, :i + 1].mean(0), atol=1e-14)
    # decode over one position returns v; over equal scores returns the mean
    od = OL.decode_attention(r.standard_normal((1, H * d)), k[:, :1], v[:, :1], H, d)
    assert np.allclose(od[0], v[0, 0], atol=1e-14)
    od = OL.decode_attention(np.zeros((1, H * d)), k, v, H, d)
    assert np.allclose(od[0], v[0].mean(0), atol=1e-14)


def test_decode_attention_loop():
    r = np.random.Generator(np.random.PCG64(14))
    S, T, H, d = 2, 7, 2, 4
    q = r.standard_normal((S, H * d))
    K, V = r.standard_normal((S, T, H * d)), r.standard_normal((S, T, H * d))
    o = OL.decode_attention(q, K, V, H, d)
    for s in range(S):
        for hh in range(H):
            sl = slice(hh * d, hh * d + d)
            ref = attn_loop(tolist(q[s, sl]), tolist(K[s, :, sl]), tolist(V[s, :, sl]), d)
            assert np.allclose(o[s, sl], ref, rtol=0, atol=1e-12)


def test_topk_attention_pins():
    r = np.random.Generator(np.random.PCG64(15))
    S, T, H, d = 2, 9, 2, 4
    q = r.standard_normal((S, H * d))
    K, V = r.standard_normal((S, T, H * d)), r.standard_normal((S, T, H * d))
    # k = T: every value is loaded, the dense result
    o, _ = OL.decode_attention_topk(q, K, V, H, d, T)
    assert np.allclose(o, OL.decode_attention(q, K, V, H, d), rtol=0, atol=1e-13)
    # k = 1: the largest-score position's probability times its value
    o1, sel = OL.decode_attention_topk(q, K, V, H, d, 1)
    for s in range(S):
        for hh in range(H):
            sl = slice(hh * d, hh * d + d)
            scores = [sum(a * b for a, b in zip(q[s, sl], K[s, t, sl])) / math.sqrt(d)
                      for t in range(T)]
            t_max = max(range(T), key=lambda t: (scores[t], -t))
            z = sum(math.exp(x - scores[t_max]) for x in scores)
            assert sel[s, hh, 0] == t_max
            assert np.allclose(o1[s, sl], V[s, t_max, sl] / z, rtol=0, atol=1e-13)
    # a middle k against a pure-Python loop (sort by score, ties to the lower position)
    k = 4
    ok, selk = OL.decode_attention_topk(q, K, V, H, d, k)
    for s in range(S):
        for hh in range(H):
            sl = slice(hh * d, hh * d + d)
            scores = [sum(a * b for a, b in zip(q[s, sl], K[s, t, sl])) / math.sqrt(d)
                      for t in range(T)]
            order = sorted(range(T), key=lambda t: (-scores[t], t))[:k]
            m = max(scores)
            z = sum(math.exp(x - m) for x in scores)
            ref = [sum(math.exp(scores[t] - m) / z * V[s, t, sl][j] for t in order)
                   for j in range(d)]
            assert list(selk[s, hh]) == order
            assert np.allclose(ok[s, sl], ref, rtol=0, atol=1e-13)
    # the kept probability mass grows with k and reaches 1 at k = T
    q2 = r.standard_normal((1, H * d))
    K2, V1 = r.standard_normal((1, T, H * d)), np.ones((1, T, H * d))
    mass = [OL.decode_attention_topk(q2, K2, V1, H, d, kk)[0][0, 0] for kk in range(1, T + 1)]
    assert all(b >= a for a, b in zip(mass, mass[1:])) and abs(mass[-1] - 1) < 1e-13


def test_topk_ties_go_to_the_lower_position():
    H, d, T = 1, 4, 6
    K = np.zeros((1, T, d))          # every score equal
    V = np.arange(T * d, dtype=np.float64).reshape(1, T, d)
    o, sel = OL.decode_attention_topk(np.ones((1, d)), K, V, H, d, 2)
    assert sel[0, 0].tolist() == [0, 1]
    assert np.allclose(o[0], (V[0, 0] + V[0, 1]) / T)
    assert OL.topk_count(543) == 55 and OL.topk_count(1056) == 106 and OL.topk_count(5) == 1


def test_relu():
    assert OL.relu(np.array([-1.0, 0.0, 2.0])).tolist() == [0.0, 0.0, 2.0]


def _tiny_layer(f=128, random_affine=True):
    wl = fg_synth.WORKLOADS["tiny"].with_(h=128, H=2, d=64, f=f, s=3, n=2, g=1, m=1)
    p = fg_synth.layer_params(wl, 0, random_affine=random_affine)
    return wl, p, OL.QuantLayer(p, wl.H, wl.d, wl.ln_eps)


def layer_loop(L, wl, xs, Kc, Vc):
    """One layer on one token (pure Python) given the K/V rows it attends over."""
    v = {k: tolist(a) for k, a in L.vec.items()}
    W = {k: tolist(a) for k, a in L.w_hat.items()}
    h, H, d = wl.h, wl.H, wl.d
    a = ln_loop(xs, v["ln1_g"], v["ln1_b"], wl.ln_eps)
    qkv = matvec_loop(a, W["wqkv"], v["bqkv"])
    q = qkv[:h]
    att = []
    for hh in range(H):
        sl = slice(hh * d, hh * d + d)
        att += attn_loop(q[sl], [k[sl] for k in Kc], [vv[sl] for vv in Vc], d)
    h1 = [xi + oi for xi, oi in zip(xs, matvec_loop(att, W["wo"], v["bo"]))]
    if L.f == 0:
        return h1, qkv
    u = ln_loop(h1, v["ln2_g"], v["ln2_b"], wl.ln_eps)
    mid = [max(t, 0.0) for t in matvec_loop(u, W["w1"], v["b1"])]
    return [a_ + b_ for a_, b_ in zip(h1, matvec_loop(mid, W["w2"], v["b2"]))], qkv


@pytest.mark.parametrize("f", [128, 0])
def test_layer_prefill_and_decode_loop(f):
    wl, p, L = _tiny_layer(f)
    r = np.random.Generator(np.random.PCG64(15))
    x = r.standard_normal((1, wl.s, wl.h)).astype(np.float16)
    cache = OL.KVCache(1, wl.s + 2, wl.h)
    y = OL.layer_prefill(L, x, cache)
    h = wl.h
    # prefill: position i attends over the fp16 K/V of positions 0..i (R5)
    kv16 = []
    for i in range(wl.s):
        _, qkv = layer_loop(L, wl, tolist(x[0, i].astype(np.float64)), [[0.0] * h], [[0.0] * h])
        kv16.append((np.array(qkv[h:2 * h]).astype(np.float16).astype(np.float64).tolist(),
                     np.array(qkv[2 * h:]).astype(np.float16).astype(np.float64).tolist()))
    for i in range(wl.s):
        ref, _ = layer_loop(L, wl, tolist(x[0, i].astype(np.float64)),
                            [kv16[j][0] for j in range(i + 1)], [kv16[j][1] for j in range(i + 1)])
        assert np.allclose(y[0, i], ref, rtol=1e-10, atol=1e-10)
    # the cache holds the quantised fp16 K/V of the prompt
    kq, ka, kb = Q.quantize_g64(np.array([kv[0] for kv in kv16], np.float16))
    assert np.array_equal(cache.qk[0, :wl.s], kq)
    # decode at pos = s: attends over the dequantised cache including the new token (R5)
    xd = r.standard_normal((1, wl.h)).astype(np.float16)
    yd = OL.layer_decode(L, xd, cache, wl.s)
    _, qkv = layer_loop(L, wl, tolist(xd[0].astype(np.float64)), [[0.0] * h], [[0.0] * h])
    knew = np.array(qkv[h:2 * h]).astype(np.float16)[None]
    vnew = np.array(qkv[2 * h:]).astype(np.float16)[None]
    krows = np.concatenate([np.array([kv[0] for kv in kv16], np.float16), knew])
    vrows = np.concatenate([np.array([kv[1] for kv in kv16], np.float16), vnew])
    khat = Q.dequant_g64(*Q.quantize_g64(krows)).astype(np.float64)
    vhat = Q.dequant_g64(*Q.quantize_g64(vrows)).astype(np.float64)
    ref, _ = layer_loop(L, wl, tolist(xd[0].astype(np.float64)), tolist(khat), tolist(vhat))
    assert np.allclose(yd[0], ref, rtol=1e-10, atol=1e-10)


def test_run_stack_positions():
    wl = fg_synth.WORKLOADS["tiny"].with_(h=128, H=2, d=64, f=128, s=4, n=3, g=1, m=2, L=2)
    layers = [OL.QuantLayer(fg_synth.layer_params(wl, l, True), wl.H, wl.d) for l in range(wl.L)]
    xp = fg_synth.prompt_states(wl)
    xs = fg_synth.step_states(wl)
    out = OL.run_stack(layers, xp, xs, cap=wl.cap)
    assert out["prefill"].shape == (wl.B, wl.s, wl.h)
    assert out["steps"].shape == (wl.n - 1, wl.B, wl.h)
    for c in out["caches"]:
        assert c.length == wl.s + wl.n - 1          # prefill + (n-1) appended tokens
    # sequences are independent: the stack over one sequence equals its row in the block
    one = OL.run_stack(layers, xp[1:2], xs[:, 1:2], cap=wl.cap)
    assert np.allclose(one["steps"][:, 0], out["steps"][:, 1], rtol=0, atol=1e-12)


def test_planted_layer_mistakes_are_caught():
    """A dropped residual or a missing 1/sqrt(d) in the oracle breaks the loop pin."""
    wl, p, L = _tiny_layer(128)
    r = np.random.Generator(np.random.PCG64(16))
    x = r.standard_normal((1, wl.s, wl.h)).astype(np.float16)
    good = OL.layer_prefill(L, x, OL.KVCache(1, wl.s, wl.h))
    orig = OL.causal_attention
    try:
        OL.causal_attention = (lambda q, k, v, H, d, dt=np.float64:
                               orig(np.asarray(q) * np.sqrt(d), k, v, H, d, dt))
        bad = OL.layer_prefill(L, x, OL.KVCache(1, wl.s, wl.h))
    finally:
        OL.causal_attention = orig
    assert not np.allclose(good, bad, rtol=1e-6, atol=1e-6)
    orig_mlp = OL._mlp_and_residual
    try:
        OL._mlp_and_residual = lambda L_, h1, dt: orig_mlp(L_, h1, dt) - h1
        bad = OL.layer_prefill(L, x, OL.KVCache(1, wl.s, wl.h))
    finally:
        OL._mlp_and_residual = orig_mlp
    assert not np.allclose(good, bad, rtol=1e-6, atol=1e-6)


# ----------------------------------------------------------------------------- the stack


def stack_loop(layers, wl, xp, xs):
    """The generation loop in pure Python, one sequence and one token at a time: prefill
    runs layer l over the prompt rows that layer l-1 produced; decode step t feeds
    x_steps[t-1] to layer 0 and each layer's output to the next, at cache length
    s + t - 1; each layer keeps its own K/V rows (fp16 in prefill, the restored 4-bit
    cache in decode) (FlexGen paper explainer, "Compute Schedule" and Algorithm 1: every
    layer over the block, then the next layer; readings R5, R9, R10)."""
    S_, s, h = xp.shape
    zero = [[0.0] * h]
    prefill = [[None] * s for _ in range(S_)]
    steps = [[None] * S_ for _ in range(xs.shape[0])]
    for b in range(S_):
        rows16 = [[] for _ in layers]          # per layer: fp16 (k, v) rows by position
        ys = [tolist(xp[b, i]) for i in range(s)]
        for l, L in enumerate(layers):
            for i in range(s):
                _, qkv = layer_loop(L, wl, ys[i], zero, zero)
                rows16[l].append((np.array(qkv[h:2 * h]).astype(np.float16),
                                  np.array(qkv[2 * h:]).astype(np.float16)))
            K = [r[0].astype(np.float64).tolist() for r in rows16[l]]
            V = [r[1].astype(np.float64).tolist() for r in rows16[l]]
            ys = [layer_loop(L, wl, ys[i], K[:i + 1], V[:i + 1])[0] for i in range(s)]
        prefill[b] = ys
        for t in range(1, xs.shape[0] + 1):
            y = tolist(xs[t - 1, b])
            for l, L in enumerate(layers):
                _, qkv = layer_loop(L, wl, y, zero, zero)
                rows16[l].append((np.array(qkv[h:2 * h]).astype(np.float16),
                                  np.array(qkv[2 * h:]).astype(np.float16)))
                assert len(rows16[l]) == s + t           # positions 0 .. s+t-1
                khat = Q.dequant_g64(*Q.quantize_g64(np.stack([r[0] for r in rows16[l]])))
                vhat = Q.dequant_g64(*Q.quantize_g64(np.stack([r[1] for r in rows16[l]])))
                y, _ = layer_loop(L, wl, y, tolist(khat), tolist(vhat))
            steps[t - 1][b] = y
    return np.array(prefill), np.array(steps)


def _stack_case():
    wl = fg_synth.WORKLOADS["tiny"].with_(h=128, H=2, d=64, f=128, s=3, n=3, g=1, m=2, L=2)
    layers = [OL.QuantLayer(fg_synth.layer_params(wl, l, True), wl.H, wl.d, wl.ln_eps)
              for l in range(wl.L)]
    return wl, layers, fg_synth.prompt_states(wl), fg_synth.step_states(wl)


def test_run_stack_matches_pure_python_loop():
    wl, layers, xp, xs = _stack_case()
    assert xs.shape[0] == 2 and len(layers) == 2
    out = OL.run_stack(layers, xp, xs, cap=wl.cap)
    pre, st = stack_loop(layers, wl, xp, xs)
    assert np.allclose(out["prefill"], pre, rtol=1e-10, atol=1e-10)
    assert np.allclose(out["steps"], st, rtol=1e-10, atol=1e-10)
    # the layers differ, so a stack that ran one of them twice would not agree
    assert not np.allclose(layers[0].w_hat["wqkv"], layers[1].w_hat["wqkv"])


def test_planted_stack_mistakes_are_caught():
    """Mistakes planted in the oracle's loop (on the CPU) that the pure-Python loop must
    catch: every layer fed the stack's input instead of the previous layer's output, and
    decode appending one position too far."""
    wl, layers, xp, xs = _stack_case()
    pre, st = stack_loop(layers, wl, xp, xs)

    orig_pre, orig_dec = OL.layer_prefill, OL.layer_decode
    first = {}

    def pre_fed_input(L, x, cache, dt=np.float64):
        if L is layers[0]:
            first["p"] = x
        return orig_pre(L, first["p"], cache, dt)

    def dec_fed_input(L, x, cache, pos, dt=np.float64):
        if L is layers[0]:
            first["d"] = x
        return orig_dec(L, first["d"], cache, pos, dt)

    def dec_shifted(L, x, cache, pos, dt=np.float64):
        return orig_dec(L, x, cache, pos + 1, dt)

    try:
        OL.layer_prefill = pre_fed_input
        bad = OL.run_stack(layers, xp, xs, cap=wl.cap + 1)
        assert not np.allclose(bad["prefill"], pre, rtol=1e-6, atol=1e-6)
        OL.layer_prefill = orig_pre
        OL.layer_decode = dec_fed_input
        bad = OL.run_stack(layers, xp, xs, cap=wl.cap + 1)
        assert np.allclose(bad["prefill"], pre, rtol=1e-10, atol=1e-10)
        assert not np.allclose(bad["steps"], st, rtol=1e-6, atol=1e-6)
        OL.layer_decode = dec_shifted
        bad = OL.run_stack(layers, xp, xs, cap=wl.cap + 1)
        assert not np.allclose(bad["steps"], st, rtol=1e-6, atol=1e-6)
    finally:
        OL.layer_prefill, OL.layer_decode = orig_pre, orig_dec
