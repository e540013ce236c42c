"""Algorithmic bytes and flops of the hot path (host logic, no GPU).

The byte formulas restate FlexGen's cost model (FlexGen paper explainer, "Cost Model
and Policy Search"): FP16 weights of one layer are 8*h1^2 + 4*h1*h2 bytes (four h1 x h1
attention matrices and two h1 x h2 MLP matrices at 2 bytes), the KV cache of one layer
is 4*bls*(s + n/2)*h1 bytes on average over decoding (keys and values at 2 bytes), and
activations are 2*bls*h1 bytes.  Under 4-bit group-wise compression every stored
element costs half a byte plus one fp16 (a, b) pair per group of 64
(FlexGen review, jaehun.me, section "4-bit 압축은 정수 연산 가속과 같은가").

These figures are what the roofline fractions in the benchmark divide by a measured
kernel time: bytes the method must move (or flops it must do), not bytes a particular
kernel happens to move.
"""
from __future__ import annotations

GROUP = 64
Q4_BYTES_PER_ELEM = 0.5 + 4.0 / GROUP          # 0.5625: codes plus (a, b) per 64


def q4_bytes(elements: float) -> float:
    return elements * Q4_BYTES_PER_ELEM


def layer_weight_elems(h: int, f: int) -> int:
    """Elements of one layer's weights: Wq, Wk, Wv, Wo (h x h) and W1, W2 (h x f)."""
    return 4 * h * h + 2 * h * f


def fp16_layer_weight_bytes(h1: int, h2: int) -> int:
    """The cost model's 8*h1^2 + 4*h1*h2."""
    return 2 * layer_weight_elems(h1, h2)


def kv_cache_bytes(layers: int, batch: int, seq: int, h: int, bytes_per_elem: float = 2.0) -> float:
    """Keys and values of ``layers`` layers for ``batch`` sequences of length ``seq``."""
    return 2.0 * layers * batch * seq * h * bytes_per_elem


def kv_cache_bytes_avg_decode(bls: int, s: int, n: int, h1: int) -> float:
    """The cost model's per-layer average over decoding, 4*bls*(s + n/2)*h1 (FP16)."""
    return 4.0 * bls * (s + n / 2.0) * h1


def weight_traffic(layers: int, layer_bytes: float, gpu_batches: int, block_reuse: bool) -> float:
    """Weight bytes loaded for one pass over ``layers`` layers by ``gpu_batches`` GPU
    batches: reloaded per batch (row-by-row) or once per block (zig-zag block)."""
    return layers * layer_bytes * (1 if block_reuse else gpu_batches)


def delegation_io_ratio(b: int, s: int, h1: int) -> float:
    """KV bytes moved for GPU attention over activation bytes moved for CPU attention:
    (b*s*h1*4) / (b*h1*4) = s."""
    return (b * s * h1 * 4.0) / (b * h1 * 4.0)


# ---------------------------------------------------------------- per-kernel work


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K


def gemm_bytes(M: int, N: int, K: int) -> float:
    """X (fp16) in, packed INT4 weights in, Y (fp16) out."""
    return 2.0 * M * K + q4_bytes(K * N) + 2.0 * M * N


def quantize_bytes(elements: float) -> float:
    """fp16 in, codes plus group statistics out."""
    return elements * (2.0 + Q4_BYTES_PER_ELEM)


def decode_attn_bytes(B: int, length: int, h: int) -> float:
    """INT4 K and V of ``length`` positions for B sequences, plus q in and out (fp16)."""
    return 2.0 * q4_bytes(B * length * h) + 4.0 * B * h


def decode_attn_topk_bytes(B: int, H: int, length: int, k: int, h: int) -> float:
    """Top-K decode attention: the whole INT4 K, the INT4 V of the k kept positions per
    head, a 4-byte score key written and read back per position and head, q in and out."""
    return (q4_bytes(B * length * h) + q4_bytes(B * k * h) + 8.0 * B * H * length
            + 4.0 * B * h)


def decode_attn_flops(B: int, length: int, h: int) -> float:
    return 4.0 * B * length * h


def prefill_attn_flops(nseq: int, s: int, h: int) -> float:
    """Causal: QK^T and PV over the lower triangle, 2 * 2 * nseq * h * s(s+1)/2."""
    return 2.0 * nseq * h * s * (s + 1)


def layernorm_bytes(rows: int, h: int) -> float:
    return 4.0 * rows * h
