"""FlexGen's analytical cost model as a throughput predictor for one GB300 (host logic).

The pages' model [FlexGen paper explainer, "Cost Model and Policy Search", "Analytical Cost
Model"] estimates one block as

    T = T_pre * l + T_gen * (n - 1) * l

with T_pre (one layer of prefill) and T_gen (one layer of one decoding step, at the average
cache length s + n/2) each the maximum over the paths that overlap: CPU<->GPU and disk<->CPU
traffic, each path's bytes summed over tensor types and divided by its bandwidth, and the
computation.  On one GB300 every tensor is resident in HBM, so the PCIe and disk paths carry no
bytes; the paths left are the HBM stream and the tensor cores.  Two granularities:

* ``"layer"`` -- the pages' form: a layer's HBM bytes over the HBM bandwidth against its
  flops over the tensor peak, assuming the two overlap perfectly across the whole layer;
* ``"kernel"`` -- the same max taken per kernel and summed, which is how a single stream of
  kernels runs (no overlap between kernels).  At the measured peaks this is the roofline-ideal
  time of the hot path.

Bytes and flops come from ``accounting`` (the method's algorithmic work: 4-bit weights and KV
at 0.5625 byte per element, fp16 activations).  The predictor ranks configurations and bounds
the measured throughput from above; it is not fitted to measurements.
"""
from __future__ import annotations

import dataclasses
import json
import os
from typing import Dict, List, Tuple

from . import accounting as A


@dataclasses.dataclass(frozen=True)
class Hardware:
    hbm_bytes_per_s: float          # copy bandwidth of HBM
    tensor_flops: float             # dense fp16 / bf16 tensor throughput

    @staticmethod
    def from_measured(path: str) -> "Hardware":
        """The measured peaks: HBM copy GB/s and the sustained bf16 GEMM rate (fp16
        runs at the bf16 rate)."""
        d = json.load(open(path))
        return Hardware(d["hbm_gbs"] * 1e9, d["bf16_tflops_sustained"] * 1e12)


@dataclasses.dataclass(frozen=True)
class Op:
    name: str
    bytes: float
    flops: float


def layer_ops(h: int, f: int, H: int, rows: int, nseq: int, kv_len: float, phase: str,
              include_aux: bool = True) -> List[Op]:
    """Kernels of one pre-LN OPT layer over ``rows`` token rows.

    phase "prefill": rows = nseq * s (causal attention over the fp16 K/V of the prompt);
    phase "decode": rows = nseq (one token per sequence, attention over ``kv_len`` cached
    positions).  ``include_aux`` adds LayerNorm and the KV quantise-append."""
    ops: List[Op] = []
    if include_aux:
        ops.append(Op("layernorm1", A.layernorm_bytes(rows, h), 0.0))
    ops.append(Op("qkv", A.gemm_bytes(rows, 3 * h, h), A.gemm_flops(rows, 3 * h, h)))
    if include_aux:
        ops.append(Op("kv_append", A.quantize_bytes(2.0 * rows * h), 0.0))
    if phase == "prefill":
        s = rows // nseq
        ops.append(Op("attention", 2.0 * 4 * rows * h, A.prefill_attn_flops(nseq, s, h)))
    else:
        ops.append(Op("attention", A.decode_attn_bytes(nseq, kv_len, h),
                      A.decode_attn_flops(nseq, kv_len, h)))
    # O projection and FC2 also read the residual row they add
    ops.append(Op("o_proj", A.gemm_bytes(rows, h, h) + 2.0 * rows * h, A.gemm_flops(rows, h, h)))
    if f > 0:
        if include_aux:
            ops.append(Op("layernorm2", A.layernorm_bytes(rows, h), 0.0))
        ops.append(Op("fc1", A.gemm_bytes(rows, f, h), A.gemm_flops(rows, f, h)))
        ops.append(Op("fc2", A.gemm_bytes(rows, h, f) + 2.0 * rows * h, A.gemm_flops(rows, h, f)))
    return ops


def phase_time(ops: List[Op], hw: Hardware, granularity: str) -> float:
    """Seconds for one layer-phase: the max over the two on-device paths, either over the
    whole layer ("layer") or per kernel and summed ("kernel")."""
    if granularity == "layer":
        return max(sum(o.bytes for o in ops) / hw.hbm_bytes_per_s,
                   sum(o.flops for o in ops) / hw.tensor_flops)
    if granularity == "kernel":
        return sum(max(o.bytes / hw.hbm_bytes_per_s, o.flops / hw.tensor_flops) for o in ops)
    raise ValueError(granularity)


def block_time(T_pre: float, T_gen: float, layers: int, n: int) -> float:
    """The pages' T = T_pre * l + T_gen * (n - 1) * l."""
    return T_pre * layers + T_gen * (n - 1) * layers


def predict(wl, hw: Hardware, granularity: str = "kernel", include_aux: bool = True) -> Dict:
    """Predicted generation throughput of a workload (fg_synth.Workload fields: h, H, f, L,
    g, m, s, n, layer_scale).  Prefill runs every layer over the whole block (B = g * m
    sequences); each decoding step attends over the average cache length s + n/2."""
    B = wl.g * wl.m
    pre = layer_ops(wl.h, wl.f, wl.H, B * wl.s, B, wl.s, "prefill", include_aux)
    gen = layer_ops(wl.h, wl.f, wl.H, B, B, wl.s + wl.n / 2.0, "decode", include_aux)
    T_pre = phase_time(pre, hw, granularity)
    T_gen = phase_time(gen, hw, granularity)
    T = block_time(T_pre, T_gen, wl.L, wl.n) * getattr(wl, "layer_scale", 1.0)
    return {"T_pre_s": T_pre, "T_gen_s": T_gen, "T_block_s": T,
            "tokens_per_s": B * wl.n / T, "granularity": granularity,
            "include_aux": include_aux}


def bottlenecks(wl, hw: Hardware) -> Dict[str, List[Tuple[str, str, float]]]:
    """Per kernel of each phase: which path bounds it and its roofline time (seconds)."""
    B = wl.g * wl.m
    out = {}
    for phase, ops in (("prefill", layer_ops(wl.h, wl.f, wl.H, B * wl.s, B, wl.s, "prefill")),
                       ("decode", layer_ops(wl.h, wl.f, wl.H, B, B, wl.s + wl.n / 2.0,
                                            "decode"))):
        rows = []
        for o in ops:
            tb, tf = o.bytes / hw.hbm_bytes_per_s, o.flops / hw.tensor_flops
            rows.append((o.name, "hbm" if tb >= tf else "tensor", max(tb, tf)))
        out[phase] = rows
    return out


def measured_peaks(root: str) -> Hardware:
    p = os.path.join(root, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return Hardware.from_measured(p)
    return Hardware(6.8e12, 1.7e15)          # one earlier measurement on a GB300
