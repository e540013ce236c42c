"""Seeded synthetic inputs and workload presets for the INT4 group-compressed OPT layer.

This module is shared by the CPU oracle (``oracle/``), the tests and ``bench.py``.
It draws random numbers and describes shapes; it holds none of the method's
arithmetic (no quantisation, no layer math).

Workloads follow the FlexGen evaluation setup (FlexGen paper explainer,
"Experimental setup" and Table 2 as summarised on the review pages): OPT-style
decoder layers, prompt 512 (or 1024) tokens, 32 generated tokens, dummy weights.
The effective batch is B = g*m: g sequences per GPU batch, m GPU batches per block
(FlexGen review, jaehun.me, section "Block은 여러 GPU 배치에 걸친 가중치 재사용 단위다").

Draws: ``numpy.random.Generator(PCG64(SeedSequence([config_id, layer, tensor_id])))``,
float32 normal, rounded to float16 nearest-even.  Weights are stored K-major with the
output channel N contiguous, i.e. ``W[K][N]`` (the transpose of torch's ``[out][in]``),
so that a group of 64 along the output channel is 64 contiguous elements.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    h: int          # hidden size
    H: int          # attention heads
    d: int          # head dim (h = H*d)
    f: int          # FFN width (0 = attention block only, no FFN)
    L: int          # decoder layers held on the device
    g: int          # sequences per GPU batch
    m: int          # GPU batches per block
    s: int          # prompt length
    n: int          # generated tokens per sequence
    outlier_frac: float = 0.0   # fraction of input channels scaled before quantisation
    outlier_scale: float = 1.0
    layer_scale: float = 1.0    # reported time is multiplied by this (8 resident of 96 layers)
    ln_eps: float = 1e-5

    @property
    def B(self) -> int:
        return self.g * self.m

    @property
    def cap(self) -> int:
        """KV cache capacity per sequence: prompt plus generated tokens."""
        return self.s + self.n

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 0, h=256, H=4, d=64, f=1024, L=2, g=2, m=2, s=16, n=4),
    "opt-6.7b": Workload("opt-6.7b", 1, h=4096, H=32, d=128, f=16384, L=4, g=16, m=4,
                         s=512, n=32),
    "opt-30b": Workload("opt-30b", 2, h=7168, H=56, d=128, f=28672, L=4, g=48, m=3,
                        s=512, n=32, outlier_frac=0.01, outlier_scale=8.0),
    "opt-175b": Workload("opt-175b", 3, h=12288, H=96, d=128, f=49152, L=8, g=36, m=4,
                         s=512, n=32, layer_scale=96.0 / 8.0),
    "kv-decode": Workload("kv-decode", 4, h=7168, H=56, d=128, f=0, L=2, g=128, m=4,
                          s=1024, n=32),
}

# tensor ids for seeding
T_WQ, T_WK, T_WV, T_WO, T_W1, T_W2 = 0, 1, 2, 3, 4, 5
T_BQKV, T_BO, T_B1, T_B2, T_LN1G, T_LN1B, T_LN2G, T_LN2B = 6, 7, 8, 9, 10, 11, 12, 13
T_OUTLIER = 20
T_XPROMPT, T_XSTEP = 100, 101
WEIGHT_STD = 0.02


def rng(config_id: int, layer: int, tensor_id: int, extra: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        [int(config_id), int(layer), int(tensor_id), int(extra)])))


def normal_fp16(shape, std: float, config_id: int, layer: int, tensor_id: int,
                extra: int = 0) -> np.ndarray:
    r = rng(config_id, layer, tensor_id, extra)
    x = r.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x.astype(np.float16)


def weight_fp16(K: int, N: int, wl: Workload, layer: int, tensor_id: int) -> np.ndarray:
    """A weight matrix W[K][N] ~ N(0, 0.02), with the workload's outlier input channels
    (a seeded subset of rows k, ``outlier_frac`` of K) scaled before fp16 rounding."""
    r = rng(wl.config_id, layer, tensor_id)
    w = r.standard_normal(size=(K, N), dtype=np.float32) * np.float32(WEIGHT_STD)
    if wl.outlier_frac > 0.0:
        k_out = max(1, int(round(wl.outlier_frac * K)))
        ro = rng(wl.config_id, layer, T_OUTLIER, tensor_id)
        rows = ro.choice(K, size=k_out, replace=False)
        w[rows, :] *= np.float32(wl.outlier_scale)
    return w.astype(np.float16)


def layer_params(wl: Workload, layer: int, random_affine: bool = False) -> Dict[str, np.ndarray]:
    """fp16 parameters of one decoder layer.

    Weights: ``wqkv`` [h][3h] (columns q | k | v), ``wo`` [h][h], ``w1`` [h][f], ``w2`` [f][h].
    Biases and LayerNorm affine are 0 / 1 / 0 (the workloads' definition) unless
    ``random_affine`` is set, which draws them so that tests exercise every term.
    """
    h, f = wl.h, wl.f
    p: Dict[str, np.ndarray] = {}
    p["wqkv"] = np.concatenate([weight_fp16(h, h, wl, layer, T_WQ),
                                weight_fp16(h, h, wl, layer, T_WK),
                                weight_fp16(h, h, wl, layer, T_WV)], axis=1)
    p["wo"] = weight_fp16(h, h, wl, layer, T_WO)
    if f > 0:
        p["w1"] = weight_fp16(h, f, wl, layer, T_W1)
        p["w2"] = weight_fp16(f, h, wl, layer, T_W2)

    def vec(n, tid, mean, std):
        if not random_affine:
            return np.full((n,), mean, dtype=np.float16)
        return (normal_fp16((n,), 1.0, wl.config_id, layer, tid).astype(np.float32)
                * np.float32(std) + np.float32(mean)).astype(np.float16)

    p["bqkv"] = vec(3 * h, T_BQKV, 0.0, 0.1)
    p["bo"] = vec(h, T_BO, 0.0, 0.1)
    p["ln1_g"] = vec(h, T_LN1G, 1.0, 0.1)
    p["ln1_b"] = vec(h, T_LN1B, 0.0, 0.1)
    p["ln2_g"] = vec(h, T_LN2G, 1.0, 0.1)
    p["ln2_b"] = vec(h, T_LN2B, 0.0, 0.1)
    if f > 0:
        p["b1"] = vec(f, T_B1, 0.0, 0.1)
        p["b2"] = vec(h, T_B2, 0.0, 0.1)
    return p


def prompt_states(wl: Workload, seqs: Optional[np.ndarray] = None) -> np.ndarray:
    """Prompt hidden states x[B][s][h] ~ N(0,1) fp16; one stream per sequence so that a
    sample of sequences can be drawn without drawing the whole block."""
    seqs = np.arange(wl.B) if seqs is None else np.asarray(seqs)
    out = np.empty((len(seqs), wl.s, wl.h), dtype=np.float16)
    for i, b in enumerate(seqs):
        out[i] = normal_fp16((wl.s, wl.h), 1.0, wl.config_id, 0, T_XPROMPT, int(b))
    return out


def step_states(wl: Workload, seqs: Optional[np.ndarray] = None) -> np.ndarray:
    """Decode-step inputs x[n-1][B][h] ~ N(0,1) fp16: a fresh hidden state per
    (step, sequence), since the layer stack has no embedding table or LM head."""
    seqs = np.arange(wl.B) if seqs is None else np.asarray(seqs)
    out = np.empty((max(wl.n - 1, 0), len(seqs), wl.h), dtype=np.float16)
    for i, b in enumerate(seqs):
        out[:, i, :] = normal_fp16((max(wl.n - 1, 0), wl.h), 1.0, wl.config_id, 0,
                                   T_XSTEP, int(b))
    return out


def sample_sequences(wl: Workload) -> np.ndarray:
    """Sequences the oracle checks at large workloads: all of them when B <= 4, else the
    first sequence of the first GPU batch and the last sequence of the last one."""
    if wl.B <= 4:
        return np.arange(wl.B)
    return np.array([0, wl.B - 1])


def adversarial_groups_fp16(seed: int = 7) -> np.ndarray:
    """Rows of 64 fp16 values that stress the group quantiser: constant groups, +-0,
    two-valued groups, values on rounding ties, the fp16 extremes, subnormals and a
    single outlier.  Returns an array [R][64] float16."""
    r = np.random.Generator(np.random.PCG64(seed))
    rows = []
    rows.append(np.full(64, 1.5, dtype=np.float16))                  # constant
    rows.append(np.full(64, -0.0, dtype=np.float16))                 # constant -0
    z = np.zeros(64, dtype=np.float16); z[::2] = -0.0; rows.append(z)   # +0 / -0 mix
    t = np.zeros(64, dtype=np.float16); t[1::2] = 3.0; rows.append(t)   # two-valued
    ties = np.array([0.0, 15.0] + [k + 0.5 for k in range(15)] * 5, dtype=np.float32)[:64]
    rows.append(ties.astype(np.float16))                             # exact half-integers
    rows.append(np.linspace(-65504, 65504, 64).astype(np.float16))   # fp16 extremes
    sub = (np.arange(64) * np.float32(2.0 ** -24)).astype(np.float16)
    rows.append(sub)                                                 # subnormals
    o = (r.standard_normal(64).astype(np.float32) * np.float32(0.02)); o[17] = 8.0
    rows.append(o.astype(np.float16))                                # single outlier
    for _ in range(8):
        rows.append((r.standard_normal(64).astype(np.float32)
                     * np.float32(10.0 ** r.uniform(-6, 4))).astype(np.float16))
    return np.stack(rows)


def random_fp16(shape, seed: int, scale: float = 1.0, offset: float = 0.0) -> np.ndarray:
    """Generic seeded N(offset, scale) fp16 array for kernel-level tests."""
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([9000, int(seed)])))
    x = r.standard_normal(size=shape, dtype=np.float32) * np.float32(scale) + np.float32(offset)
    return x.astype(np.float16)


def random_q4_cache_torch(B: int, H: int, cap: int, d: int, seed: int, device="cuda"):
    """Seeded random contents of one layer's 4-bit KV cache, drawn on the device with
    torch (for workloads too large to draw on the host): codes uniform in 0..15 packed two
    per byte, group minimum a ~ N(0, 1) and maximum b = a + |N(0, 2)|, stored as the fp16
    bit pairs (a low, b high).  Returns (k_codes, v_codes, k_ab, v_ab) shaped like the
    library's cache: [B][H][cap][d/2] uint8 and [B][H][cap][d/64] int32."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = []
    for _ in range(2):
        codes = torch.randint(0, 256, (B, H, cap, d // 2), generator=g, device=device,
                              dtype=torch.int32).to(torch.uint8)
        out.append(codes)
    for _ in range(2):
        a = torch.randn((B, H, cap, d // 64), generator=g, device=device)
        b = a + torch.randn((B, H, cap, d // 64), generator=g, device=device).abs() * 2.0
        ab = (a.half().view(torch.int16).to(torch.int32) & 0xFFFF) | \
             (b.half().view(torch.int16).to(torch.int32) << 16)
        out.append(ab)
    return out[0], out[1], out[2], out[3]
