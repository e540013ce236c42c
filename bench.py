"""Generated tokens/s of an OPT-shaped INT4 layer stack on one or more GB300s.

One step = one whole generation pass over the block: prefill of every layer over the
prompt of all B = g*m sequences, then n-1 decode steps each running every layer over the
whole block (FlexGen's block schedule).  tokens per step = B * n (the prefill yields the
first token; FlexGen paper explainer, "Analytical Cost Model": T = Tpre*l + Tgen*(n-1)*l;
throughput = generated tokens / (prefill + decode) time, FlexGen review (jaehun.me)).

Default workload: the OPT-175B-shaped stack, the largest configuration that fits one GPU
(hidden 12288, 96 heads x 128, FFN 49152, B = 144 = 36 x 4, prompt 512, 32 generated
tokens), 8 layers resident with the time scaled by 96/8 to the whole stack, weights
N(0, 0.02) and KV cache in 4-bit groups of 64; inputs are seeded synthetic hidden states
N(0, 1).  The other workloads (OPT-6.7B, OPT-30B and the KV-dominated decode) run after
it for a few steps each and are reported under ``per_config``; the KV-dominated one gives
the metric's second half, decode-attention HBM GB/s as a fraction of peak.

`value` times K steps replayed from one CUDA graph (inputs resident in HBM); per-kernel
roofline figures come from eager passes (prefill and decode apart) with CUDA events around
every launch.  `e2e` times K steps with every step's inputs copied from pinned host memory
and its generated hidden states copied back inside the timed region, the copies of
neighbouring steps overlapping the compute on their own streams.  `--impl reference` and
`cpu_baseline` time the CPU oracle on a bounded sample of the same workload.

Multi-GPU (torchrun): every rank runs its own block of sequences (sequences never
interact, so there is no data-path collective); `value` is all ranks' tokens over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fg_synth  # noqa: E402
from bit_compressed_throughput_gb300 import replicas  # noqa: E402

METRIC = "generated tokens/s per OPT-shaped layer stack at 1 GB300; decode-attn HBM GB/s % peak"
UNIT = "tokens/s"
DEFAULT_CONFIG = "opt-175b"
SUB_CONFIGS = ("opt-6.7b", "opt-30b", "kv-decode")
# Nominal GB300 figures (context for the measured-peak fractions): HBM3e 7.9 TB/s, dense
# fp16/bf16 tensor 2.25 PFLOP/s
NOMINAL_HBM_GBS = 7900.0
NOMINAL_F16_TFLOPS = 2250.0
# DRAM bytes (read + write) per launch of the prefill GEMM, by workload: from one-kernel ncu
# captures (dram__bytes_read.sum + dram__bytes_write.sum, one pass) at full size, averaged over
# one pass's launch mix; a workload without a capture of the current kernel reports null.
# opt-175b: the QKV, O, FC1 and FC2 projections of one GPU batch (18432 tokens, equal launch
# counts per pass) in the fp16-weight mode of the layer prefill (profile case
# layer-prefill-opt175b), units in dynamic order, read + wrote 16.16, 6.77, 21.46 and
# 42.12 GB; their algorithmic bytes (X, the fp16 weights, Y, and the residual read of O and
# FC2) are 2.72, 1.66, 3.47 and 3.93 GB.
GEMM_TRAFFIC_PER_LAUNCH = {"opt-175b": 21629349376}
GEMM_ALGORITHMIC_BYTES_PER_LAUNCH = {"opt-175b": 2944401408}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def workload_desc(wl):
    scale = getattr(wl, "layer_scale", 1.0)
    tail = (f", time x{scale:g} for the whole stack ({wl.L} layers run)" if scale != 1.0 else "")
    return (f"{wl.name}: h{wl.h} H{wl.H}x{wl.d} f{wl.f} L{wl.L} B{wl.B} (g{wl.g} m{wl.m}) "
            f"s{wl.s} n{wl.n}, int4 g64 weights + KV, fp16 compute{tail}")


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for nm, v in zip(names, r[5:9]):
                    if v.strip() == "Active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm


def build_stack(wl, device, seed_offset=0):
    """Quantised layers and a block of inputs, generated on the device (seeded)."""
    import torch
    from bit_compressed_throughput_gb300 import fg
    g = torch.Generator(device=device)
    layers = []
    for l in range(wl.L):
        g.manual_seed(1000 * wl.config_id + l)
        params = {}
        for name, K, N in (("wqkv", wl.h, 3 * wl.h), ("wo", wl.h, wl.h),
                           ("w1", wl.h, wl.f), ("w2", wl.f, wl.h)):
            if N == 0 or K == 0:
                continue
            w = torch.randn((K, N), generator=g, device=device) * fg_synth.WEIGHT_STD
            if wl.outlier_frac > 0:
                rows = torch.randperm(K, generator=g, device=device)[:max(1, int(round(
                    wl.outlier_frac * K)))]
                w[rows] *= wl.outlier_scale
            params[name] = w.half()
            del w
        h, f = wl.h, wl.f
        params.update({"bqkv": torch.zeros(3 * h), "bo": torch.zeros(h), "ln1_g": torch.ones(h),
                       "ln1_b": torch.zeros(h), "ln2_g": torch.ones(h), "ln2_b": torch.zeros(h)})
        if f:
            params.update({"b1": torch.zeros(f), "b2": torch.zeros(h)})
        layers.append(fg.LayerQ4.from_fp16(params, wl.H, wl.ln_eps, device=device))
        del params
    g.manual_seed(77 + seed_offset)
    x = torch.randn((wl.B, wl.s, wl.h), generator=g, device=device).half()
    xs = torch.randn((max(wl.n - 1, 1), wl.B, wl.h), generator=g, device=device).half()
    torch.cuda.synchronize()
    return layers, x, xs


class Runner:
    """Fixed device buffers for one generation pass, runnable eagerly or from a graph."""

    def __init__(self, wl, layers, x, xs, device):
        import torch
        from bit_compressed_throughput_gb300 import fg
        self.fg, self.wl = fg, wl
        self.eng = fg.StackEngine(layers, wl.g, wl.m, wl.cap, wl.s, device=device)
        self.x, self.xs = x, xs
        self.y = torch.empty_like(x)                                   # prefill output
        self.out = torch.empty((max(wl.n - 1, 1), wl.B, wl.h), dtype=torch.float16,
                               device=device)                          # decode outputs
        self.graph = None

    def prefill(self):
        self.eng.prefill(self.x, self.y, self.wl.s)

    def decode_all(self):
        wl = self.wl
        for t in range(1, wl.n):
            self.eng.decode(self.xs[t - 1], self.out[t - 1], wl.s + t - 1)

    def step(self):
        self.prefill()
        self.decode_all()

    def capture(self):
        import torch
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()


def time_region(fn, steps, dist=None):
    import torch
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        fn()
    e1.record(st)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return replicas.max_over_ranks(e0.elapsed_time(e1), dist, device="cuda")


def time_e2e_pipelined(runs, hx, hxs, hout, hlast, steps, dist=None):
    """Milliseconds for `steps` generation passes through the public path with host I/O:
    step i's inputs are copied from pinned host memory (copy-in stream), its graph replays
    once they have landed (compute stream), and its outputs (the decode states and the
    prefill's last position) are copied back (copy-out stream).  Step i uses buffer set
    i % 2, so step i+1's inputs and step i-1's outputs move while step i computes; a set is
    refilled only after the graph that read it finished, and its outputs are overwritten
    only after they were copied out.  The region ends when the last outputs reached the
    host."""
    import torch
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    done = [None, None]            # graph of the set finished (inputs free, outputs ready)
    out_free = [None, None]        # outputs of the set copied to the host
    in_ready = [None, None]

    def copy_in(i):
        r = runs[i % 2]
        with torch.cuda.stream(cin):
            if done[i % 2] is not None:
                cin.wait_event(done[i % 2])
            r.x.copy_(hx, non_blocking=True)
            r.xs.copy_(hxs, non_blocking=True)
            in_ready[i % 2] = torch.cuda.Event()
            in_ready[i % 2].record(cin)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    cin.wait_stream(comp)
    cout.wait_stream(comp)
    copy_in(0)
    for i in range(steps):
        k = i % 2
        r = runs[k]
        if i + 1 < steps:
            copy_in(i + 1)
        comp.wait_event(in_ready[k])
        if out_free[k] is not None:
            comp.wait_event(out_free[k])
        r.replay()
        done[k] = torch.cuda.Event()
        done[k].record(comp)
        with torch.cuda.stream(cout):
            cout.wait_event(done[k])
            hlast.copy_(r.y[:, -1, :], non_blocking=True)
            hout.copy_(r.out, non_blocking=True)
            out_free[k] = torch.cuda.Event()
            out_free[k].record(cout)
    comp.wait_stream(cout)
    e1.record(comp)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return replicas.max_over_ranks(e0.elapsed_time(e1), dist, device="cuda")


def cost_model_line(wl, value):
    """The pages' analytical cost model re-parameterised with the measured peaks: the
    roofline-ideal throughput of this workload and the measured fraction of it."""
    from bit_compressed_throughput_gb300 import cost_model
    hw = cost_model.measured_peaks(ROOT)
    p = cost_model.predict(wl, hw, "kernel", include_aux=True)
    return {"predicted_tokens_per_s": round(p["tokens_per_s"], 1),
            "measured_over_predicted": round(value / p["tokens_per_s"], 4),
            "granularity": "per-kernel max(HBM bytes / bandwidth, flops / tensor peak), summed",
            "peaks": "measured HBM copy and sustained bf16"}


def profile_phase(fg, fn, steps):
    """Per-kernel launches, milliseconds and algorithmic work of `steps` eager runs of fn
    (CUDA events around every launch on its stream)."""
    fg.fg_prof_reset()
    fg.fg_prof_enable(True)
    ms = time_region(fn, steps)
    fg.fg_prof_enable(False)
    return ms, {fg.KINDS[k]: fg.fg_prof_query(k) for k in range(len(fg.KINDS))}


def roof(kernel, p, pk, bound, steps, extra=None):
    """Roofline entry of one kernel kind from its profile record: achieved = algorithmic
    work / event time, against the measured peak (copy bandwidth, or sustained bf16 for a
    kernel timed inside a long pass) and against the nominal one."""
    if not p or not p["launches"] or not p["ms"]:
        return None
    if bound == "hbm":
        a, unit, peak, nom = p["work"] / (p["ms"] * 1e-3) / 1e9, "GB/s", pk["hbm_gbs"], \
            NOMINAL_HBM_GBS
        src = f"{pk['source']} HBM copy"
    else:
        a, unit, peak, nom = p["work"] / (p["ms"] * 1e-3) / 1e12, "TFLOP/s", \
            pk["bf16_sustained"], NOMINAL_F16_TFLOPS
        src = f"{pk['source']} bf16 sustained (fp16 dense rate equal)"
    r = {"kernel": kernel, "bound": bound, "achieved": round(a, 1), "peak": peak, "unit": unit,
         "frac": round(a / peak, 4), "peak_source": src, "peak_nominal": nom,
         "frac_of_nominal": round(a / nom, 4), "launches_per_step": p["launches"] // steps,
         "ms_per_step": round(p["ms"] / steps, 3)}
    if extra:
        r.update(extra)
    return r


def kernel_table(prof, steps):
    return {k: {"launches_per_step": v["launches"] // steps, "ms_per_step": round(v["ms"] / steps, 3)}
            for k, v in prof.items() if v["launches"]}


TENSOR_GEMMS = ("gemm_f16w_pair", "q4_dequant_gemm_pair", "q4_dequant_gemm_tc")


def merged_gemm(prof):
    """The tensor-bound GEMM launches of a phase (CTA-pair and one-CTA tiled kernels) as one
    record, named by the kinds that ran."""
    kinds = [k for k in TENSOR_GEMMS if prof[k]["launches"]]
    rec = {f: sum(prof[k][f] for k in kinds) for f in ("launches", "ms", "work")}
    return "+".join(kinds) or TENSOR_GEMMS[0], rec


def prefill_attn_roof(wl, rec, pk, steps):
    """Causal prefill attention against the roof that binds at its arithmetic intensity: a
    launch reads Q, K and V (3h fp16 columns per token of its g sequences) and writes the
    output (h columns), 8*g*s*h bytes, for 2*g*h*s*(s+1) flops.  At s = 512 that is s/4 = 128
    flop per byte, below the ridge of the measured peaks (~265), so the HBM floor is the
    higher one; the tensor fraction is reported beside it."""
    if not rec or not rec["launches"] or not rec["ms"]:
        return None
    nbytes = 8.0 * wl.g * wl.s * wl.h * rec["launches"]
    flops = rec["work"]
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_sustained"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    tensor = roof("prefill_attn", rec, pk, "tensor", steps)
    if bound == "tensor":
        r = tensor
    else:
        r = roof("prefill_attn", dict(rec, work=nbytes), pk, "hbm", steps)
        r["tensor_frac"] = tensor["frac"]
        r["tensor_achieved_tflops"] = tensor["achieved"]
    r["flop_per_byte"] = round(flops / nbytes, 1)
    r["ridge_flop_per_byte"] = round(pk["bf16_sustained"] * 1e12 / (pk["hbm_gbs"] * 1e9), 1)
    r["bytes_per_launch"] = int(8 * wl.g * wl.s * wl.h)
    return r


def phase_rooflines(wl, pre, dec, pk, psteps):
    """Rooflines of the prefill and decode kernels of one workload."""
    pname, prec = merged_gemm(pre)
    out = {"prefill_gemm": roof(pname, prec, pk, "tensor", psteps),
           "prefill_attn": prefill_attn_roof(wl, pre["prefill_attn"], pk, psteps),
           "decode_attn": roof("q4kv_decode_attn", dec["q4kv_decode_attn"], pk, "hbm", psteps,
                               {"lengths": f"{wl.s + 1}..{wl.s + wl.n - 1}",
                                "sequences_x_heads": wl.B * wl.H})}
    ds = dec["q4_dequant_gemm_stream"]
    dname, drec = merged_gemm(dec)
    if ds["launches"]:
        out["decode_gemm"] = roof("q4_dequant_gemm_stream", ds, pk, "hbm", psteps,
                                  {"M": wl.B, "kernel_kind": "weight-streaming (M <= 128)"})
    if drec["launches"]:
        # M = B tokens: 3.56*M flop per weight byte, above the ridge for M >= 144
        wb = 0.5625 * (4 * wl.h * wl.h + 2 * wl.h * wl.f) * wl.L * (wl.n - 1) * psteps
        out["decode_gemm"] = roof(dname, drec, pk, "tensor", psteps,
                                  {"M": wl.B, "kernel_kind": "tiled (M > 128)",
                                   "weight_gbs": round(wb / (drec["ms"] * 1e-3) / 1e9, 1)})
    return out


def fused_gemm_probe(fg, wl, layer, device, pk, reps=3):
    """The dequant-fused GEMM (4-bit codes restored inside the mainloop, C-ABI
    fg_dequant_gemm_q4) at this workload's prefill FC1 shape (QKV without an FFN), timed
    alone with CUDA events.  The layer's prefill restores each layer's weights once and runs
    the fp16-weight mode of the same kernel instead; this line keeps the fused kernel
    measured at the prefill shape."""
    import torch
    W, epi = (layer.w1, 1) if wl.f else (layer.wqkv, 0)
    M, K, N = wl.g * wl.s, W.K, W.N
    gen = torch.Generator(device=device)
    gen.manual_seed(11)
    X = torch.randn((M, K), generator=gen, device=device).half()
    Y = torch.empty((M, N), dtype=torch.float16, device=device)
    bias = torch.zeros(N, dtype=torch.float16, device=device)
    wsb = fg.fg_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(wsb, dtype=torch.uint8, device=device) if wsb else None
    fg.fg_dequant_gemm_q4(X, W, bias, epi, None, Y, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fg.fg_dequant_gemm_q4(X, W, bias, epi, None, Y, ws)
    e1.record()
    torch.cuda.synchronize()
    fg.fg_check_device_error()
    ms = e0.elapsed_time(e1) / reps
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    del X, Y, ws
    return {"kernel": "q4_dequant_gemm_pair", "shape": f"M={M} K={K} N={N}", "bound": "tensor",
            "achieved": round(tf, 1), "unit": "TFLOP/s", "ms_per_launch": round(ms, 3),
            "peak": pk["bf16"], "frac": round(tf / pk["bf16"], 4),
            "frac_of_sustained": round(tf / pk["bf16_sustained"], 4),
            "peak_source": f"{pk['source']} bf16 burst (timed alone, {reps} launches)",
            "frac_of_nominal": round(tf / NOMINAL_F16_TFLOPS, 4)}


def run_config(wl, device, steps, warmup, dist=None, rank=0, full=False, pk=None):
    """Build one workload's stack on the device and time it: the graph-replayed pass,
    eager per-kernel profiles of prefill and decode, and (full) the e2e pass with host I/O."""
    import torch
    from bit_compressed_throughput_gb300 import fg
    layers, x, xs = build_stack(wl, device, seed_offset=rank)
    run = Runner(wl, layers, x, xs, device)
    for _ in range(warmup):
        run.step()
    torch.cuda.synchronize()
    fg.fg_check_device_error()
    run.capture()
    run.replay()
    torch.cuda.synchronize()

    clk = ClockSampler(torch.cuda.current_device())
    ms = time_region(run.replay, steps, dist)
    clocks = clk.stop()
    fg.fg_check_device_error()

    psteps = max(1, min(steps, 3))
    ms_pre, pre = profile_phase(fg, run.prefill, psteps)
    ms_dec, dec = profile_phase(fg, run.decode_all, psteps)
    launches_per_step = (sum(p["launches"] for p in pre.values())
                         + sum(p["launches"] for p in dec.values())) // psteps
    scale = getattr(wl, "layer_scale", 1.0)
    world = dist.get_world_size() if dist is not None else 1
    value = replicas.total_tokens(world, wl.B, wl.n, steps) / (ms * 1e-3 * scale)
    res = {"workload": workload_desc(wl), "value": round(value, 2), "unit": UNIT,
           "ms_per_step": round(ms / steps, 3), "steps": steps, "warmup": warmup,
           "eager_ms_per_step": {"prefill": round(ms_pre / psteps, 3),
                                 "decode": round(ms_dec / psteps, 3)},
           "rooflines": phase_rooflines(wl, pre, dec, pk, psteps),
           "kernels": {"prefill": kernel_table(pre, psteps), "decode": kernel_table(dec, psteps)},
           "cost_model": cost_model_line(wl, value),
           "gpu_launches_per_step": launches_per_step, "clocks": clocks}
    extra = {"pre": pre, "psteps": psteps}

    if full:
        # end to end: every step's inputs copied in from pinned host memory and its generated
        # hidden states copied back, inside the region; two buffer sets (each with its own
        # engine and graph) let step i+1's inputs and step i's outputs move on copy streams
        # while step i computes
        hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        hxs = torch.empty(xs.shape, dtype=xs.dtype, pin_memory=True)
        hx.copy_(x)
        hxs.copy_(xs)
        hout = torch.empty(run.out.shape, dtype=run.out.dtype, pin_memory=True)
        hlast = torch.empty((wl.B, wl.h), dtype=torch.float16, pin_memory=True)
        run_b = Runner(wl, layers, torch.empty_like(x), torch.empty_like(xs), device)
        run_b.step()
        torch.cuda.synchronize()
        run_b.capture()
        ms_e2e = time_e2e_pipelined([run, run_b], hx, hxs, hout, hlast, steps, dist)
        extra["e2e"] = {
            "value": round(replicas.total_tokens(world, wl.B, wl.n, steps)
                           / (ms_e2e * 1e-3 * scale), 2),
            "unit": UNIT, "h2d_bytes_per_step": (hx.numel() + hxs.numel()) * 2,
            "d2h_bytes_per_step": (hout.numel() + hlast.numel()) * 2,
            "copies": "every step's inputs in and outputs out on copy streams, overlapped "
                      "with the neighbouring steps' compute (two buffer sets)"}
        del run_b
        extra["fused_prefill_gemm"] = fused_gemm_probe(fg, wl, layers[0], device, pk)
    del run, layers, x, xs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res, extra


def run_gpu(args, wl):
    import torch
    world, rank, local = dist_env()
    dist = None
    # the CPU baseline's oracle set-up (weight draws and quantisation, one host core) runs
    # in a child process while the GPU works; its timed sample runs after the GPU part
    child = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        child = subprocess.Popen([sys.executable, os.path.abspath(__file__), "--oracle-child",
                                  "--config", wl.name], stdin=subprocess.PIPE,
                                 stdout=subprocess.PIPE, text=True)
    if world > 1:
        import torch.distributed as D
        torch.cuda.set_device(local)
        D.init_process_group("nccl")
        dist = D
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    import __graft_entry__
    __graft_entry__.build()

    pk = peaks()
    main, extra = run_config(wl, device, args.steps, args.warmup, dist, rank, full=True, pk=pk)
    per_config = {}
    if not args.no_sub_configs and world == 1:
        for name in SUB_CONFIGS:
            if name == wl.name:
                continue
            sub, _ = run_config(fg_synth.WORKLOADS[name], device, min(args.steps, 5), 3, None,
                                rank, full=False, pk=pk)
            per_config[name] = sub

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None
    rl = main["rooflines"]
    gemm = dict(rl["prefill_gemm"]) if rl["prefill_gemm"] else {}
    if gemm:
        gemm.pop("ms_per_step", None)
        gemm["traffic"] = GEMM_TRAFFIC_PER_LAUNCH.get(wl.name)
        gemm["traffic_note"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch "
                                "(mean of the four prefill projection shapes, fp16-weight mode); "
                                "the weights are re-read from HBM per raster group of token "
                                "tiles and when the clusters sharing a k-block drift apart"
                                if gemm["traffic"] else
                                "no one-kernel capture of the current GEMM at this workload")
        if gemm["traffic"]:
            gemm["algorithmic_bytes_per_launch"] = GEMM_ALGORITHMIC_BYTES_PER_LAUNCH[wl.name]
        gemm["share_of_kernel_time"] = round(
            merged_gemm(extra["pre"])[1]["ms"] / extra["psteps"]
            / max(1e-9, main["eager_ms_per_step"]["prefill"] + main["eager_ms_per_step"]["decode"]),
            4)
    kvw = per_config.get("kv-decode", main if wl.name == "kv-decode" else None)
    attn_kv = kvw["rooflines"]["decode_attn"] if kvw else None
    res = {
        "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) hidden states, N(0,0.02) weights, random init)",
        "config": {"workload": main["workload"], "tokens_per_step": wl.B * wl.n,
                   "parallelism": f"replicas x{world} (one block of B={wl.B} per GPU)",
                   "graph": "one CUDA graph per generation pass",
                   "l2": "no flush: per-step working set (4-bit weights "
                         f"{wl.L * 0.5625 * (4 * wl.h * wl.h + 2 * wl.h * wl.f) / 1e6:.0f} MB, "
                         f"KV {wl.L * 2 * 0.5625 * wl.B * wl.cap * wl.h / 1e6:.0f} MB, "
                         f"prompt {wl.B * wl.s * wl.h * 2 / 1e6:.0f} MB) exceeds the 129 MB L2"},
        "roofline": gemm or None,
        "decode_gemm_roofline": rl.get("decode_gemm"),
        "decode_attn_roofline": rl["decode_attn"],
        "decode_attn_hbm_kv_workload": attn_kv,
        "prefill_attn_roofline": rl["prefill_attn"],
        "dequant_fused_prefill_gemm": extra.get("fused_prefill_gemm"),
        "kernels": main["kernels"],
        "cost_model": main["cost_model"],
        "eager_ms_per_step": main["eager_ms_per_step"],
        "gpu_launches": main["gpu_launches_per_step"] * args.steps,
        "e2e": extra["e2e"],
        "clocks": main["clocks"],
        "per_config": per_config,
    }
    if child is not None:
        res["cpu_baseline"] = finish_oracle_child(child)
    if dist is not None:
        dist.destroy_process_group()
    return res


# ----------------------------------------------------------------------------- CPU oracle


def oracle_setup(wl, n_layers):
    import oracle
    params = [fg_synth.layer_params(wl, l) for l in range(n_layers)]
    return [oracle.QuantLayer(p, wl.H, wl.d, wl.ln_eps, keep_codes=False) for p in params]


def oracle_sample(wl, layer, seq: int):
    """One sequence through one layer: the prefill over the prompt, then the first decode
    step.  Returns (seconds of the prefill, seconds of the decode step)."""
    import oracle
    xp = fg_synth.prompt_states(wl, np.array([seq]))
    xs = fg_synth.step_states(wl, np.array([seq]))
    cache = oracle.KVCache(1, wl.cap, wl.h)
    t0 = time.perf_counter()
    oracle.layer_prefill(layer, xp, cache, np.float32)
    t1 = time.perf_counter()
    oracle.layer_decode(layer, xs[0], cache, wl.s, np.float32)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def oracle_tokens_per_s(wl, t_pre, t_dec):
    """Throughput of the stack from one sequence-layer sample, by the pages' cost model
    T = Tpre*l + Tgen*(n-1)*l (FlexGen paper explainer, "Analytical Cost Model"): the
    oracle's decode step costs the same at every cache length of these workloads (its time
    is the weight products), so one decode step stands for each of the n-1."""
    per_seq_stack = (t_pre + (wl.n - 1) * t_dec) * wl.L * getattr(wl, "layer_scale", 1.0)
    return wl.n / per_seq_stack


SAMPLE_DESC = ("1 sequence x 1 layer of {name}: the prefill over the {s}-token prompt and the "
               "first decode step, numpy float32, BLAS threads default; tokens/s = n / ((Tpre + "
               "(n-1)*Tdec) x {L} layers{scale}) (the pages' cost model)")


def sample_desc(wl):
    sc = getattr(wl, "layer_scale", 1.0)
    return SAMPLE_DESC.format(name=wl.name, s=wl.s, L=wl.L,
                              scale=f" x {sc:g}" if sc != 1.0 else "")


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count()


def oracle_child(wl):
    """Child process of the GPU arm: builds the oracle's quantised layer, says "ready",
    waits for a line on stdin (sent once the GPU part is done), times one sample and
    prints it as JSON."""
    layer = oracle_setup(wl, 1)[0]
    print("ready", flush=True)
    sys.stdin.readline()
    t_pre, t_dec = oracle_sample(wl, layer, 0)
    print(json.dumps({"t_pre": t_pre, "t_dec": t_dec}), flush=True)


def finish_oracle_child(child):
    """Tells the child to time its sample and returns its (t_pre, t_dec) record."""
    out, _ = child.communicate("go\n", timeout=1800)
    lines = [ln for ln in out.strip().splitlines() if ln.startswith("{")]
    if child.returncode != 0 or not lines:
        return {"value": None, "unit": UNIT, "kind": "oracle", "error": "oracle child failed"}
    return json.loads(lines[-1])


def cpu_baseline_line(wl, d):
    v = oracle_tokens_per_s(wl, d["t_pre"], d["t_dec"])
    return {"value": round(v, 5), "unit": UNIT, "cores": cores(), "kind": "oracle",
            "sample": sample_desc(wl), "sample_seconds": round(d["t_pre"] + d["t_dec"], 3)}


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    layer = oracle_setup(wl, 1)[0]
    for i in range(args.warmup):
        oracle_sample(wl, layer, i)
    pre, dec = [], []
    t0 = time.perf_counter()
    for i in range(args.steps):
        a, b = oracle_sample(wl, layer, args.warmup + i)
        pre.append(a)
        dec.append(b)
    wall = time.perf_counter() - t0
    value = oracle_tokens_per_s(wl, statistics.mean(pre), statistics.mean(dec))
    cb = {"value": round(value, 5), "unit": UNIT, "cores": cores(), "kind": "oracle",
          "sample": "each step: " + sample_desc(wl)}
    return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall / args.steps * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)", "config": {"workload": workload_desc(wl)},
            "sample_scaling": "ms_per_step is the measured time of one step's sample; value "
                              "scales it to the workload by the cost model stated in "
                              "cpu_baseline.sample",
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(fg_synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-configs", action="store_true",
                    help="time only --config (skip the other workloads' per_config lines)")
    ap.add_argument("--oracle-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    wl = fg_synth.WORKLOADS[args.config]
    if args.oracle_child:
        oracle_child(wl)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        res = run_reference(args, wl)
    else:
        res = run_gpu(args, wl)
        if res is not None and isinstance(res.get("cpu_baseline"), dict) \
                and "t_pre" in res["cpu_baseline"]:
            res["cpu_baseline"] = cpu_baseline_line(wl, res["cpu_baseline"])
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
