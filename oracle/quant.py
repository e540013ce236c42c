"""Group-wise asymmetric 4-bit quantisation (oracle).  Test infrastructure only.

Source: FlexGen review (jaehun.me), section "4-bit 압축은 정수 연산 가속과 같은가"
(restating paper §5): weights and KV cache are stored as 4-bit integers and restored
to FP16 before compute; weights are grouped 64 elements at a time along the output
channel, the KV cache along the hidden dimension; quantisation is asymmetric with
the group minimum ``a`` and maximum ``b``; recovery is not exact and a constant group
(a == b) needs its own handling.  "论文阅读：FlexGen" (blog.gzher.com) §3.4 adds that
the scheme is fine-grained group-wise asymmetric quantisation, kept low-bit in
storage and dequantised to FP16 before compute.

The pages lose the formula itself.  Readings taken where they are silent or garbled:

R1  code  q = round((x - a) * 15 / (b - a)), evaluated in IEEE binary32, one rounding per
    operation, in this order: xf = float(x); d = xf - af; t = d * 15; r = t / (b - a);
    q = rint(r) (round half to even); q = clamp(q, 0, 15).
R2  a, b are the group minimum and maximum of the fp16 values (exact, stored as fp16).
    Ties between -0 and +0 are broken by the total order -0 < +0.
R3  constant group (b - a == 0): every code is 0.
R4  dequant  x^ = fp16_rn(a + q * ((b - a) / 15)), in binary32: s = (b - a) / 15;
    p = q * s; x32 = a + p; round to fp16 nearest-even.
RP  packing: element 2i in the low nibble and element 2i+1 in the high nibble of byte i,
    along the grouped (contiguous) dimension.

numpy's float32 ufuncs are IEEE binary32 operations with round-to-nearest-even and
no contraction across separate ufunc calls, which is what R1 and R4 require.
"""
from __future__ import annotations

import numpy as np

GROUP = 64
QMAX = 15


def _order_key(bits: np.ndarray) -> np.ndarray:
    """Map fp16 bit patterns to unsigned keys whose order is the numeric order of the
    values, with -0 < +0 (reading R2).  NaN is outside the contract."""
    u = bits.astype(np.uint32)
    neg = (u & 0x8000) != 0
    return np.where(neg, 0x7FFF - (u & 0x7FFF), 0x8000 + u).astype(np.uint32)


def group_min_max(x: np.ndarray):
    """Per-group minimum a and maximum b of an fp16 array [R][C] (C % 64 == 0),
    groups of 64 consecutive elements along the last axis.  Returns fp16 arrays
    [R][C/64]."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    R, C = x.shape
    assert C % GROUP == 0, "grouped dimension must be a multiple of 64"
    xg = x.reshape(R, C // GROUP, GROUP)
    key = _order_key(xg.view(np.uint16))
    ia = key.argmin(axis=-1)[..., None]
    ib = key.argmax(axis=-1)[..., None]
    a = np.take_along_axis(xg, ia, axis=-1)[..., 0]
    b = np.take_along_axis(xg, ib, axis=-1)[..., 0]
    return a, b


def quantize_g64(x: np.ndarray):
    """Quantise fp16 x[R][C] group-wise (64 along C) to 4-bit codes (R1-R3).

    Returns (q, a, b): q uint8 [R][C] with values 0..15 (unpacked), a and b fp16
    [R][C/64].  Parity: pinned (closed-form ties, exact binary32 emulation with
    fractions, invariants)."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    R, C = x.shape
    a, b = group_min_max(x)
    af = a.astype(np.float32)
    bf = b.astype(np.float32)
    bma = bf - af                                     # binary32, one rounding
    xf = x.reshape(R, C // GROUP, GROUP).astype(np.float32)   # exact
    d = xf - af[..., None]
    t = d * np.float32(QMAX)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = t / bma[..., None]
    q = np.rint(r)                                    # round half to even
    q = np.clip(q, 0, QMAX)
    const = (bma == 0)[..., None]                     # R3
    q = np.where(const, 0.0, q)
    return q.astype(np.uint8).reshape(R, C), a, b


def dequant_g64(q: np.ndarray, a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Restore fp16 values from codes q[R][C] (unpacked) and group stats a, b [R][C/64]
    by R4.  Parity: pinned (exact binary32 emulation, constant groups, error bound)."""
    R, C = q.shape
    af = a.astype(np.float32)[..., None]
    bf = b.astype(np.float32)[..., None]
    s = (bf - af) / np.float32(QMAX)
    p = q.reshape(R, C // GROUP, GROUP).astype(np.float32) * s
    x32 = af + p
    return x32.astype(np.float16).reshape(R, C)


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """RP: byte i holds element 2i (low nibble) and 2i+1 (high nibble)."""
    q = np.asarray(q, dtype=np.uint8)
    assert q.shape[-1] % 2 == 0
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 0x0F
    out[..., 1::2] = codes >> 4
    return out


def ab_pack_u32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Storage form of the group statistics: one 32-bit word per group, a's fp16 bits
    in the low half and b's in the high half."""
    return (a.astype(np.float16).view(np.uint16).astype(np.uint32)
            | (b.astype(np.float16).view(np.uint16).astype(np.uint32) << 16))
