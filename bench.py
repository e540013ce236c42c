"""Generated tokens/s of an OPT-shaped INT4 layer stack on one or more GB300s.

One step = one whole generation pass over the block: prefill of every layer over the
prompt of all B = g*m sequences, then n-1 decode steps each running every layer over the
whole block (FlexGen's block schedule).  tokens per step = B * n (the prefill yields the
first token; FlexGen paper explainer, "Analytical Cost Model": T = Tpre*l + Tgen*(n-1)*l;
throughput = generated tokens / (prefill + decode) time, FlexGen review (jaehun.me)).

Default workload: OPT-6.7B-shaped stack (hidden 4096, 32 heads x 128, FFN 16384, 4
layers, B = 64 = 16 x 4, prompt 512, 32 generated tokens), weights N(0, 0.02) and KV
cache in 4-bit groups of 64.  Inputs are seeded synthetic hidden states N(0, 1).

`value` times K steps replayed from one CUDA graph (inputs resident in HBM);
per-kernel roofline figures come from an eager pass over the same K steps with CUDA
events around every launch.  `e2e` times the same K steps with every step's inputs copied from
pinned host memory and its generated hidden states copied back inside the timed region, the
copies of neighbouring steps overlapping the compute on their own streams.
`--impl reference` times the CPU oracle on a bounded sample of the same workload.

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
# DRAM bytes (read + write) per launch of the tiled GEMM (the prefill GEMMs; decode runs the
# streaming kernel): the mean over its 64 launches in one generation pass of this workload,
# from an ncu capture of dram__bytes_read.sum and dram__bytes_write.sum; reset to None
# whenever the GEMM kernel changes
GEMM_TRAFFIC_PER_LAUNCH = 501274876


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

    def step(self):
        wl = self.wl
        self.eng.prefill(self.x, self.y, wl.s)
        for t in range(1, wl.n):
            self.eng.decode(self.xs[t - 1], self.out[t - 1], wl.s + t - 1)

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


def run_gpu(args, wl):
    import torch
    world, rank, local = dist_env()
    dist = None
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
    from bit_compressed_throughput_gb300 import fg

    layers, x, xs = build_stack(wl, device, seed_offset=rank)
    run = Runner(wl, layers, x, xs, device)
    for _ in range(args.warmup):
        run.step()
    torch.cuda.synchronize()
    fg.fg_check_device_error()
    run.capture()
    run.replay()
    torch.cuda.synchronize()

    tokens_per_step = wl.B * wl.n
    clk = ClockSampler(torch.cuda.current_device())
    ms = time_region(run.replay, args.steps, dist)
    clocks = clk.stop()
    fg.fg_check_device_error()

    # eager pass over the same K steps with per-launch events (roofline figures)
    fg.fg_prof_reset()
    fg.fg_prof_enable(True)
    ms_eager = time_region(run.step, args.steps, dist)
    fg.fg_prof_enable(False)
    prof = {fg.KINDS[k]: fg.fg_prof_query(k) for k in range(len(fg.KINDS))}
    launches = sum(p["launches"] for p in prof.values())

    # end to end: every step's inputs copied in from pinned host memory and its generated
    # hidden states copied back, inside the region; two buffer sets (each with its own
    # engine and graph) let step i+1's inputs and step i's outputs move on copy streams while
    # step i computes
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
    ms_e2e = time_e2e_pipelined([run, run_b], hx, hxs, hout, hlast, args.steps, dist)
    h2d = (hx.numel() + hxs.numel()) * 2
    d2h = (hout.numel() + hlast.numel()) * 2

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None
    pk = peaks()
    g_ = prof["q4_dequant_gemm_tc"]
    gemm_tflops = g_["work"] / (g_["ms"] * 1e-3) / 1e12 if g_["ms"] else None
    d_ = prof["q4_dequant_gemm_stream"]
    dgemm_gbs = d_["work"] / (d_["ms"] * 1e-3) / 1e9 if d_["ms"] else None
    a_ = prof["q4kv_decode_attn"]
    attn_gbs = a_["work"] / (a_["ms"] * 1e-3) / 1e9 if a_["ms"] else None
    total_kernel_ms = sum(p["ms"] for p in prof.values())
    # a workload that keeps a slice of its layers resident reports its time scaled to the
    # whole stack (the 175B shape: 8 of 96 layers, time x 96/8)
    scale = getattr(wl, "layer_scale", 1.0)
    value = replicas.total_tokens(world, wl.B, wl.n, args.steps) / (ms * 1e-3 * scale)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) hidden states, N(0,0.02) weights, random init)",
        "config": {"workload": workload_desc(wl), "tokens_per_step": tokens_per_step,
                   "parallelism": f"replicas x{world} (one block of B={wl.B} per GPU)",
                   "graph": "one CUDA graph per generation pass",
                   "l2": "no flush: per-step working set (4-bit weights "
                         f"{wl.L * 0.5625 * (4 * wl.h * wl.h + 2 * wl.h * wl.f) / 1e6:.0f} MB, "
                         f"KV {wl.L * 2 * 0.5625 * wl.B * wl.cap * wl.h / 1e6:.0f} MB, "
                         f"prompt {wl.B * wl.s * wl.h * 2 / 1e6:.0f} MB) exceeds the 129 MB L2"},
        "roofline": {"kernel": "q4_dequant_gemm_tc", "bound": "tensor",
                     "achieved": round(gemm_tflops, 1) if gemm_tflops else None,
                     "peak": pk["bf16_sustained"], "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / pk["bf16_sustained"], 4) if gemm_tflops else None,
                     "peak_source": f"{pk['source']} bf16 sustained (fp16 dense rate equal)",
                     "traffic": GEMM_TRAFFIC_PER_LAUNCH,
                     "share_of_kernel_time": round(g_["ms"] / total_kernel_ms, 4)
                     if total_kernel_ms else None},
        "decode_gemm_roofline": {"kernel": "q4_dequant_gemm_stream", "bound": "hbm",
                                 "achieved": round(dgemm_gbs, 1) if dgemm_gbs else None,
                                 "peak": pk["hbm_gbs"], "unit": "GB/s",
                                 "frac": round(dgemm_gbs / pk["hbm_gbs"], 4) if dgemm_gbs else None,
                                 "launches": d_["launches"]},
        "decode_attn_roofline": {"kernel": "q4kv_decode_attn", "bound": "hbm",
                                 "achieved": round(attn_gbs, 1) if attn_gbs else None,
                                 "peak": pk["hbm_gbs"], "unit": "GB/s",
                                 "frac": round(attn_gbs / pk["hbm_gbs"], 4) if attn_gbs else None,
                                 "launches": a_["launches"]},
        "kernels": {k: {"launches": v["launches"], "ms": round(v["ms"], 3)}
                    for k, v in prof.items() if v["launches"]},
        "cost_model": cost_model_line(wl, value),
        "eager_ms_per_step": round(ms_eager / args.steps, 3),
        "gpu_launches": launches,
        "e2e": {"value": round(replicas.total_tokens(world, wl.B, wl.n, args.steps)
                               / (ms_e2e * 1e-3 * scale), 2),
                "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "every step's inputs in and outputs out on copy streams, overlapped "
                          "with the neighbouring steps' compute (two buffer sets)"},
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, samples=1)
    if dist is not None:
        dist.destroy_process_group()
    return res


# ----------------------------------------------------------------------------- CPU oracle


def oracle_setup(wl, n_layers):
    import oracle
    params = [fg_synth.layer_params(wl, l) for l in range(n_layers)]
    return [oracle.QuantLayer(p, wl.H, wl.d, wl.ln_eps, keep_codes=False) for p in params]


def oracle_sample_step(wl, layers, seq: int):
    """One sequence through the sampled layers: prefill over the prompt, n-1 decode
    steps.  Returns seconds."""
    import oracle
    xp = fg_synth.prompt_states(wl, np.array([seq]))
    xs = fg_synth.step_states(wl, np.array([seq]))
    t0 = time.perf_counter()
    oracle.run_stack(layers, xp, xs, cap=wl.cap, dt=np.float32)
    return time.perf_counter() - t0


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count()


def cpu_baseline(wl, samples=1):
    """The oracle (numpy, float32 products) on the host cores: one sequence through one
    layer of the workload (prefill + n-1 decode steps), scaled to the L-layer stack."""
    layers = oracle_setup(wl, 1)
    secs = [oracle_sample_step(wl, layers, s) for s in range(samples)]
    per_seq_stack = statistics.mean(secs) * wl.L * getattr(wl, "layer_scale", 1.0)
    return {"value": round(wl.n / per_seq_stack, 4), "unit": UNIT, "cores": cores(),
            "kind": "oracle",
            "sample": f"1 sequence x 1 layer of {wl.name} (prefill {wl.s} + {wl.n - 1} decode "
                      f"steps), time x{wl.L} layers; numpy float32, BLAS threads default"}


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    layers = oracle_setup(wl, 1)
    for i in range(args.warmup):
        oracle_sample_step(wl, layers, i)
    t = sum(oracle_sample_step(wl, layers, args.warmup + i) for i in range(args.steps))
    # one sequence through the L-layer stack (scaled to the whole stack as the GPU arm is)
    per_step = t / args.steps * wl.L * getattr(wl, "layer_scale", 1.0)
    value = wl.n / per_step
    cb = {"value": round(value, 4), "unit": UNIT, "cores": cores(), "kind": "oracle",
          "sample": f"each step: 1 sequence x 1 layer of {wl.name} (prefill {wl.s} + "
                    f"{wl.n - 1} decode steps), time x{wl.L} layers; numpy float32"}
    return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)", "config": {"workload": workload_desc(wl)},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default="opt-6.7b", choices=sorted(fg_synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = fg_synth.WORKLOADS[args.config]
    res = run_reference(args, wl) if args.impl == "reference" else run_gpu(args, wl)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
