"""Pins of the oracle's group-wise 4-bit quantiser against what the pages and the
mathematics fix, independently of the oracle's own code.

The pages (FlexGen review, jaehun.me, section "4-bit 압축은 정수 연산 가속과 같은가";
"论文阅读：FlexGen" §3.4) fix: 4-bit codes, groups of 64 along the output channel
(weights) or the hidden dimension (KV), asymmetric with the group min a and max b,
inexact recovery, constant groups handled on their own.  The formula itself is lost in
the page text; its reading (binary32, round half to even) is checked here by an exact
rational evaluation that rounds each operation to binary32 by hand.

Each ``check_*`` helper takes the functions under test, so the same checks are run on
the oracle (must pass) and on copies with a planted mistake (must fail).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import fg_synth
from oracle import quant as Q

# ----------------------------------------------------------------------------- exact
# rounding of a rational to an IEEE binary format (round to nearest, ties to even)


def _round_fmt(x: Fraction, p: int, emin: int) -> Fraction:
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    ax = abs(x)
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    while Fraction(2) ** e > ax:
        e -= 1
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - (p - 1))
    m = ax / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * quantum


def f32(x: Fraction) -> Fraction:
    return _round_fmt(x, 24, -126)


def f16(x: Fraction) -> Fraction:
    return _round_fmt(x, 11, -14)


def rint_even(x: Fraction) -> int:
    fl = x.numerator // x.denominator
    rem = x - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def frac(v) -> Fraction:
    return Fraction(float(v))


def exact_code(x, a, b) -> int:
    """R1 evaluated with every operation rounded to binary32 by hand."""
    xf, af, bf = frac(x), frac(a), frac(b)
    bma = f32(bf - af)
    if bma == 0:
        return 0
    d = f32(xf - af)
    t = f32(d * 15)
    r = f32(t / bma)
    return min(max(rint_even(r), 0), 15)


def exact_dequant(q, a, b) -> Fraction:
    """R4 evaluated with every operation rounded to binary32, then to binary16."""
    af, bf = frac(a), frac(b)
    s = f32(f32(bf - af) / 15)
    p = f32(q * s)
    return f16(f32(af + p))


# ----------------------------------------------------------------------------- inputs


def all_finite_fp16_sorted():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = bits.view(np.float16)
    v = v[np.isfinite(v)]
    v = np.unique(v.astype(np.float64))          # drops the duplicate zero
    return v.astype(np.float16)


def groups_from_sorted(v):
    n = (len(v) // 64) * 64
    return v[:n].reshape(-1, 64)


def random_groups(n_rows=64, seed=1):
    r = np.random.Generator(np.random.PCG64(seed))
    rows = []
    for i in range(n_rows):
        scale = 10.0 ** r.uniform(-5, 4)
        rows.append((r.standard_normal(64) * scale + r.uniform(-1, 1) * scale)
                    .astype(np.float16))
    return np.stack(rows)


# ----------------------------------------------------------------------------- checks


def check_codes_exact(quantize, x):
    q, a, b = quantize(x)
    bad = []
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            g = j // 64
            e = exact_code(x[i, j], a[i, g], b[i, g])
            if int(q[i, j]) != e:
                bad.append((i, j, float(x[i, j]), int(q[i, j]), e))
    return bad


def check_group_stats(quantize, x):
    """a, b are the min and max over 64 contiguous elements (brute force)."""
    q, a, b = quantize(x)
    bad = []
    for i in range(x.shape[0]):
        for g in range(x.shape[1] // 64):
            vals = [float(v) for v in x[i, 64 * g:64 * g + 64]]
            if float(a[i, g]) != min(vals) or float(b[i, g]) != max(vals):
                bad.append((i, g))
    return bad


def check_invariants(quantize, dequant, x):
    """codes in [0,15]; min -> 0 and max -> 15 in non-constant groups; constant groups
    are all-zero codes and recover exactly; the round-trip error bound holds."""
    q, a, b = quantize(x)
    errs = []
    if q.min() < 0 or q.max() > 15:
        errs.append("code range")
    xh = dequant(q, a, b)
    R, C = x.shape
    u = 2.0 ** -24
    for i in range(R):
        for g in range(C // 64):
            sl = slice(64 * g, 64 * g + 64)
            xs = x[i, sl].astype(np.float64)
            qs = q[i, sl]
            A, Bv = float(a[i, g]), float(b[i, g])
            if A == Bv:
                if qs.any() or not np.all(xh[i, sl].astype(np.float64) == xs):
                    errs.append(("constant", i, g))
                continue
            if qs[int(np.argmin(xs))] != 0 or qs[int(np.argmax(xs))] != 15:
                errs.append(("endpoints", i, g))
            if np.any(xs < A) or np.any(xs > Bv):
                errs.append(("a<=x<=b", i, g))
            delta = Bv - A
            xhat = xh[i, sl].astype(np.float64)
            ulp16 = _ulp16(xhat)
            bound = delta / 30 + 8 * u * delta + 2 * u * max(abs(A), abs(Bv)) + 0.5 * ulp16
            if np.any(np.abs(xs - xhat) > bound * (1 + 1e-12)):
                errs.append(("bound", i, g, float(np.max(np.abs(xs - xhat) - bound))))
    return errs


def _ulp16(v):
    """Spacing of binary16 at |v| (normal: 2^(e-10); subnormal: 2^-24)."""
    av = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(av > 0, av, 1.0)))
    return np.where(av >= 2.0 ** -14, 2.0 ** (e - 10), 2.0 ** -24)


def check_dequant_exact(dequant, q, a, b):
    xh = dequant(q, a, b)
    bad = []
    for i in range(q.shape[0]):
        for j in range(q.shape[1]):
            g = j // 64
            e = exact_dequant(int(q[i, j]), a[i, g], b[i, g])
            if Fraction(float(xh[i, j])) != e:
                bad.append((i, j))
    return bad


# ----------------------------------------------------------------------------- tests


def test_ties_round_half_even_closed_form():
    """Group with a = 0, b = 15: the code is the value itself rounded half to even, so
    0.5 -> 0, 1.5 -> 2, 2.5 -> 2, ... (closed form of R1; binary32 is exact here)."""
    vals = [0.0, 15.0] + [k + 0.5 for k in range(15)] + [float(k) for k in range(15)]
    vals = (vals * 3)[:64]
    x = np.array([vals], dtype=np.float16)
    q, a, b = Q.quantize_g64(x)
    expect = []
    for v in vals:
        fl = math.floor(v)
        if v - fl == 0.5:
            expect.append(fl if fl % 2 == 0 else fl + 1)
        else:
            expect.append(int(round(v)))
    assert [int(c) for c in q[0]] == expect
    assert float(a[0, 0]) == 0.0 and float(b[0, 0]) == 15.0


def test_codes_match_exact_binary32_all_fp16_values():
    """Every finite fp16 value, in groups of 64 consecutive sorted values and in wide
    random groups, quantised by the oracle equals R1 evaluated exactly."""
    v = all_finite_fp16_sorted()
    x = groups_from_sorted(v)
    assert check_codes_exact(Q.quantize_g64, x) == []                # all 992 groups
    assert check_codes_exact(Q.quantize_g64, random_groups(48)) == []
    assert check_codes_exact(Q.quantize_g64, fg_synth.adversarial_groups_fp16()) == []


def test_group_stats_are_min_max_of_contiguous_64():
    x = np.concatenate([random_groups(8).reshape(2, 256),
                        fg_synth.adversarial_groups_fp16()[:8].reshape(2, 256)])
    assert check_group_stats(Q.quantize_g64, x) == []


def test_minus_zero_plus_zero_order():
    x = np.zeros((1, 64), np.float16)
    x[0, 5] = np.float16(-0.0)
    q, a, b = Q.quantize_g64(x)
    assert a.view(np.uint16)[0, 0] == 0x8000 and b.view(np.uint16)[0, 0] == 0x0000
    assert not q.any()


def test_invariants_random_and_adversarial():
    for x in (random_groups(64), fg_synth.adversarial_groups_fp16(),
              groups_from_sorted(all_finite_fp16_sorted())[::31]):
        assert check_invariants(Q.quantize_g64, Q.dequant_g64, x) == []


def test_dequant_matches_exact_binary32():
    r = np.random.Generator(np.random.PCG64(3))
    x = np.concatenate([random_groups(16), fg_synth.adversarial_groups_fp16()])
    q, a, b = Q.quantize_g64(x)
    qr = r.integers(0, 16, size=q.shape).astype(np.uint8)   # codes not tied to x
    assert check_dequant_exact(Q.dequant_g64, q, a, b) == []
    assert check_dequant_exact(Q.dequant_g64, qr, a, b) == []


def test_packing_closed_form_and_round_trip():
    q = np.array([[1, 2, 3, 4, 15, 0]], np.uint8)
    assert Q.pack_nibbles(q).tolist() == [[0x21, 0x43, 0x0F]]
    r = np.random.Generator(np.random.PCG64(5)).integers(0, 16, (7, 128)).astype(np.uint8)
    assert np.array_equal(Q.unpack_nibbles(Q.pack_nibbles(r)), r)


def test_ab_storage_word():
    a = np.array([[1.0]], np.float16)
    b = np.array([[-2.0]], np.float16)
    assert int(Q.ab_pack_u32(a, b)[0, 0]) == (0xC000 << 16) | 0x3C00


def test_grouping_direction_with_outlier_input_channels():
    """Weights group along the output channel N at fixed input channel k: scaling one
    input channel (row k of W[K][N]) widens exactly that row's groups."""
    wl = fg_synth.WORKLOADS["tiny"].with_(outlier_frac=0.02, outlier_scale=8.0)
    w = fg_synth.weight_fp16(128, 256, wl, 0, fg_synth.T_WQ)
    q, a, b = Q.quantize_g64(w)
    width = (b.astype(np.float64) - a.astype(np.float64)).mean(axis=1)
    big = np.argsort(width)[-3:]
    base = np.median(width)
    assert np.all(width[big] > 4 * base)


# ------------------------------------------------------------- planted mistakes (CPU)


def _floor_quantize(x):
    q, a, b = Q.quantize_g64(x)
    af = a.astype(np.float32)[..., None]
    bf = b.astype(np.float32)[..., None]
    R, C = x.shape
    xf = x.reshape(R, C // 64, 64).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (xf - af) * np.float32(15) / (bf - af)
    qq = np.where((bf - af) == 0, 0, np.clip(np.floor(r), 0, 15))
    return qq.astype(np.uint8).reshape(R, C), a, b


def _half_away_quantize(x):
    q, a, b = Q.quantize_g64(x)
    af = a.astype(np.float32)[..., None]
    bf = b.astype(np.float32)[..., None]
    R, C = x.shape
    xf = x.reshape(R, C // 64, 64).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = ((xf - af) * np.float32(15)) / (bf - af)
    qq = np.where((bf - af) == 0, 0, np.clip(np.floor(r + np.float32(0.5)), 0, 15))
    return qq.astype(np.uint8).reshape(R, C), a, b


def _transposed_groups_quantize(x):
    q, a, b = Q.quantize_g64(np.ascontiguousarray(x.T))
    return np.ascontiguousarray(q.T), a, b   # wrong grouping axis


def _dequant_scale16(q, a, b):
    R, C = q.shape
    af = a.astype(np.float32)[..., None]
    bf = b.astype(np.float32)[..., None]
    s = (bf - af) / np.float32(16)
    return (af + q.reshape(R, C // 64, 64) * s).astype(np.float16).reshape(R, C)


def _dequant_no_offset(q, a, b):
    R, C = q.shape
    af = a.astype(np.float32)[..., None]
    bf = b.astype(np.float32)[..., None]
    s = (bf - af) / np.float32(15)
    return (q.reshape(R, C // 64, 64) * s).astype(np.float16).reshape(R, C)


def test_planted_mistakes_are_caught():
    x = random_groups(32)
    ties = np.array([[0.0, 15.0] + [k + 0.5 for k in range(15)] * 5], np.float32)[:, :64]
    ties = ties.astype(np.float16)
    assert check_invariants(_floor_quantize, Q.dequant_g64, x) != []
    assert check_codes_exact(_half_away_quantize, ties) != []
    sq = random_groups(64)
    assert check_group_stats(_transposed_groups_quantize, sq) != []
    assert check_invariants(Q.quantize_g64, _dequant_scale16, x) != []
    assert check_invariants(Q.quantize_g64, _dequant_no_offset, x) != []
