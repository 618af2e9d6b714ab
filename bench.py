"""Benchmark of the quantised MoE layer forward (decode) on GB300.

One step = one whole-layer forward (router, top-k, grouping, gate/up +
SwiGLU, down, combine + residual + shared expert) over one batch of
synthetic tokens.  Default workload: 64 experts top-2, hidden 4096, expert
intermediate 4096, INT4 group 128, Zipf(1.1) routing skew, 8 tokens per call.
Steps rotate over several layer instances (weights far larger than L2) and
over 16 token batches, so every step streams its experts from HBM.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (the only reference implementation there is).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_expert_ffn_warp_gb300 import synth  # noqa: E402

METRIC = "MoE-layer decode tokens/s and achieved HBM GB/s (% of GB300 peak) at 1 GPU"
UNIT = "tokens/s"
GATEUP_SRC = os.path.join(ROOT, "quantized_expert_ffn_warp_gb300", "csrc", "ffn.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="e64_top2_zipf")
    ap.add_argument("--n", type=int, default=None, help="tokens per call")
    ap.add_argument("--layers", type=int, default=4, help="layer instances rotated per step")
    ap.add_argument("--batches", type=int, default=16)
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of a graph")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--quick", action="store_true", help="small run for profiling")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config sub-record (every config and token count)")
    ap.add_argument("--prenorm", action="store_true",
                    help="time the layer with the two-pass RMSNorm in front "
                         "(moe_forward_prenorm on a synthetic residual stream)")
    ap.add_argument("--gemm-min-tokens", type=int, default=None,
                    help="experts with at least this many tokens use the tcgen05 GEMM kernels "
                         "(0: decode kernels only; default: the library's)")
    return ap.parse_args()


def kernels_per_forward(spec, n, info, prenorm=False):
    """Kernels one forward launches: routing (two launches on the large-batch
    route: from 64 tokens, or from 8 with at least 128 experts), grouping
    (inside the routing launch for at most 256 pairs), gate/up, down, combine;
    the gather and the two GEMM kernels when some expert can reach the GEMM
    threshold; the RMSNorm in front with --prenorm."""
    m = info["gemm_min_tokens"]
    route = 2 if n >= 64 or (spec.n_experts >= 128 and n >= 8) else 1
    group = 0 if n * spec.top_k <= 256 else 1
    gemm = 3 if spec.wbits == 4 and m > 0 and n >= m else 0
    return route + group + 3 + gemm + (1 if prenorm else 0)


def workload_name(spec, n, prenorm=False):
    s = "%s: E=%d top-%d H=%d I=%d INT%d g%d" % (spec.name, spec.n_experts, spec.top_k,
                                                 spec.hidden, spec.inter, spec.wbits, spec.group)
    if prenorm:
        s = "RMSNorm + " + s
    if spec.has_shared:
        s += " +shared(I=%d, sigmoid gate)" % spec.shared_inter
    s += ", %s routing, %d tokens/call" % (
        "Zipf(%g)" % spec.zipf_s if spec.zipf_s else "uniform", n)
    return s


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def replica_seeds(rank, n_layers):
    """Seeds of a rank's layer instances and of its token batches: every rank
    is an independent replica with its own seeded layers and tokens."""
    return [1000 * rank + i for i in range(n_layers)], rank


def max_over_ranks(pg, ms, device):
    """The slowest rank's time: the whole job finishes when it does."""
    if not pg:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput: the units every rank processed over the max time."""
    return units_per_rank * world / (ms / 1e3)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            p = [v.strip() for v in line.split(",")]
            if len(p) >= 8:
                self.rows.append(p)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


def file_hash(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def recorded_traffic(config, n):
    """DRAM bytes per gate/up launch from the committed ncu summary, if the
    kernel source is unchanged since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ffn_traffic.txt")
    if not os.path.exists(p):
        return None
    sha = file_hash(GATEUP_SRC)
    for line in open(p):
        f = line.split()
        if len(f) == 4 and not f[0].startswith("#") and f[0] == config and f[1] == str(n) \
                and f[2] == sha:
            return float(f[3])
    return None


NORM_EPS = 1e-6   # RMSNorm eps of the --prenorm workload


def cpu_oracle_rate(spec, n, seconds, layer=None, prenorm=False):
    """Tokens/s of the CPU oracle (as it stands) on a bounded sample: whole
    forwards of the same workload until `seconds` have elapsed (with the
    RMSNorm in front for --prenorm)."""
    import oracle
    oracle.build()
    if layer is None:
        layer = synth.make_layer(spec, 0)
    gain = synth.make_norm_gain(spec) if prenorm else None
    t0 = time.perf_counter()
    calls = 0
    while True:
        if prenorm:
            x = oracle.rmsnorm(synth.make_residual(spec, n, seed=0, batch=calls % 16), gain,
                               NORM_EPS)
        else:
            x = synth.make_tokens(spec, n, seed=0, batch=calls % 16)
        oracle.forward(layer, x)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds or calls >= 64:
            break
    return calls * n / el, calls, el, oracle.num_threads()


def run_reference(args, spec, n, rank, world):
    """The reference arm: the CPU oracle as it stands, exactly `warmup`
    untimed and `steps` timed steps.  A step is one whole-layer forward of n
    tokens; when one forward takes longer than the per-step share of
    --cpu-seconds, a step routes all n tokens and computes the outputs of an
    evenly spread subset, and the rate counts the tokens computed."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    layer = synth.make_layer(spec, 0)
    gain = synth.make_norm_gain(spec) if args.prenorm else None

    def tokens_of(i):
        if args.prenorm:
            return oracle.rmsnorm(synth.make_residual(spec, n, seed=0, batch=i % 16), gain,
                                  NORM_EPS)
        return synth.make_tokens(spec, n, seed=0, batch=i % 16)

    t0 = time.perf_counter()
    oracle.forward(layer, tokens_of(0))               # also the first warm-up step
    one = time.perf_counter() - t0
    budget = args.cpu_seconds / max(1, args.steps + args.warmup)
    per_step = n if one <= budget else max(1, int(n * budget / one))
    sel = None if per_step == n else np.unique(
        np.linspace(0, n - 1, per_step).round().astype(np.int32))
    per_step = n if sel is None else len(sel)
    for i in range(1, args.warmup):
        oracle.forward(layer, tokens_of(i), tokens=sel)
    xs = [tokens_of(args.warmup + i) for i in range(min(args.steps, 16))]
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.forward(layer, xs[i % len(xs)], tokens=sel)
    el = time.perf_counter() - t0
    rate = args.steps * per_step / el
    sample = ("%d whole-layer forwards of %d tokens (%.1f s)" % (args.steps, n, el)
              if sel is None else
              "%d steps, each routing %d tokens and computing the outputs of %d of them (%.1f s)"
              % (args.steps, n, per_step, el))
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(spec, n, args.prenorm), "n_tokens": n},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class StepRunner:
    """Runs steps k0 .. k0 + k - 1 of a rotation of `period` forwards: whole
    periods by one captured CUDA graph, the others by per-step graphs, so any
    step count can be run exactly (eagerly with use_graph=False)."""

    def __init__(self, step, period, st, use_graph):
        import torch
        self.step, self.period, self.st = step, period, st
        self.full, self.single = None, []
        if not use_graph:
            return
        with torch.cuda.stream(st):
            for i in range(period):       # the exact sequence once before capture
                step(i, st)
        st.synchronize()
        self.full = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            with torch.cuda.graph(self.full, stream=st):
                for i in range(period):
                    step(i, st)
            for i in range(period):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=st):
                    step(i, st)
                self.single.append(g)

    def run(self, k0, k):
        import torch
        with torch.cuda.stream(self.st):
            if self.full is None:
                for i in range(k0, k0 + k):
                    self.step(i, self.st)
                return
            i, end = k0, k0 + k
            while i < end:
                if i % self.period == 0 and end - i >= self.period:
                    self.full.replay()
                    i += self.period
                else:
                    self.single[i % self.period].replay()
                    i += 1


def timed_reps(fn, k0, K, st, pg, device, min_ms, min_steps, max_reps=10000):
    """Repetitions of exactly K steps (fn(k0, K) launches them on st), each
    timed by CUDA events on st between a barrier + synchronize on both sides;
    max over ranks per repetition.  Repeats until the timed total reaches
    min_ms and min_steps steps.  Returns (per-repetition ms, next step)."""
    import torch
    times = []
    total = 0.0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    while True:
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        e0.record(st)
        fn(k0, K)
        e1.record(st)
        e1.synchronize()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        ms = max_over_ranks(pg, e0.elapsed_time(e1), device)
        times.append(ms)
        total += ms
        k0 += K
        if (total >= min_ms and len(times) * K >= min_steps) or len(times) >= max_reps:
            return times, k0


def gate_up_bytes(spec, touched, n):
    """Algorithmic bytes of one gate/up launch: the touched experts' gate and
    up codes, scales and zeros, the shared expert's, and the activations."""
    H = spec.hidden

    def gu(inter):
        return 2 * (inter * H * spec.wbits // 8 + inter * (H // 128) * 3)
    return touched * gu(spec.inter) + (gu(spec.shared_inter) if spec.has_shared else 0) + n * H * 2


def down_bytes(spec, touched):
    H = spec.hidden

    def dn(inter):
        return H * inter * spec.wbits // 8 + H * (inter // 128) * 3
    return touched * dn(spec.inter) + (dn(spec.shared_inter) if spec.has_shared else 0)


def measure_layers(layers, xs, spec, n, st, use_graph=True, prenorm_gain=None, min_ms=60.0,
                   min_steps=32):
    """Times forwards rotating over (layer, batch) pairs; returns the median
    per-forward time, per-phase times (eager pass with events) and the
    touched experts per step, from the library's own routing."""
    import torch
    from quantized_expert_ffn_warp_gb300 import moe
    L, B = len(layers), len(xs)
    period = int(np.lcm(L, B))
    outs = [torch.empty_like(xs[0]) for _ in range(B)]

    def step(i, s):
        li, b = i % L, i % B
        if prenorm_gain is not None:
            layers[li].forward_prenorm(xs[b], prenorm_gain, NORM_EPS, outs[b], stream=s)
        else:
            layers[li].forward(xs[b], outs[b], stream=s)

    touched = []
    for i in range(period):
        x = xs[i % B]
        if prenorm_gain is not None:
            x = moe.rmsnorm(x, prenorm_gain, NORM_EPS, stream=st)
        r = layers[i % L].route_topk(x, stream=st)
        st.synchronize()
        touched.append(int((r["counts"] > 0).sum().item()))
    runner = StepRunner(step, period, st, use_graph)
    runner.run(0, period)                 # warm-up
    times, _ = timed_reps(runner.run, 0, period, st, None, None, min_ms, min_steps)
    us = 1e3 * statistics.median(times) / period
    for lay in layers:
        lay.profile_enable(True)
    with torch.cuda.stream(st):
        for i in range(period):
            step(i, st)
    st.synchronize()
    phase, calls = {p: 0.0 for p in moe.PHASES}, 0
    for lay in layers:
        d, c = lay.profile_read()
        lay.profile_enable(False)
        for p in d:
            phase[p] += d[p]
        calls += c
    phase_us = {p: 1e3 * phase[p] / max(calls, 1) for p in phase}
    return us, phase_us, float(np.mean(touched)), times


# Config, tokens per call, and whether the point is a supplementary
# tensor-bound one (large-batch GEMM beyond the configs' token counts).
CONFIG_POINTS = [("tiny", 4, False),
                 ("e256_top8_shared", 1, False), ("e256_top8_shared", 16, False),
                 ("e512_top4_shared", 1, False), ("e512_top4_shared", 4, False),
                 ("e512_top4_shared", 32, False),
                 ("e512_top4_shared_2bit", 1, False), ("e512_top4_shared_2bit", 4, False),
                 ("e512_top4_shared_2bit", 32, False)] + \
    [(c, n, False) for c in ("e64_top2_sweep", "e64_top2_sweep_zipf")
     for n in (1, 8, 64, 256, 1024)] + \
    [("e64_top2_sweep", 4096, True), ("e64_top2_sweep", 8192, True)]


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return json.load(open(p)).get("bf16_tflops", 1900.0), "measured"
    return 1900.0, "fallback"


def run_config_points(dev, st, peak, points, log=None):
    """The configs sub-record: every config and token count on seeded
    device-drawn layers (same distributions as the parity tests' layers),
    each timed as a CUDA-graph rotation over layer instances and 16 token
    batches."""
    import torch
    from quantized_expert_ffn_warp_gb300 import moe
    tflops_peak, tflops_kind = bf16_peak()
    out = []
    by_cfg = {}
    for name, n, extra in points:
        by_cfg.setdefault(name, []).append((n, extra))
    for name, pts in by_cfg.items():
        spec = synth.CONFIGS[name]
        per_layer = synth.expert_bytes(spec) * spec.n_experts + synth.expert_bytes(spec, True)
        n_layers = 2 if per_layer > 1e9 else 4
        max_n = max(n for n, _ in pts)
        layers = []
        for i in range(n_layers):
            w = synth.make_layer_device(spec, seed=100 + i, device=dev)
            layers.append(moe.MoeLayer(spec, w, max_tokens=max_n))
            del w
        torch.cuda.synchronize()
        for n, extra in pts:
            B = 16 if n <= 1024 else 4
            xs = [torch.from_numpy(synth.make_tokens(spec, n, seed=7, batch=b).view(np.float16))
                  .to(dev) for b in range(B)]
            us, ph, touched, times = measure_layers(layers, xs, spec, n, st)
            ab = synth.spec_algorithmic_bytes(spec, touched, n)
            gu = gate_up_bytes(spec, touched, n)
            dn = down_bytes(spec, touched)
            rec = {"config": name, "n": n, "us_per_forward": us, "tokens_per_s": n / (us * 1e-6),
                   "touched_experts": touched,
                   "whole_layer_frac": ab / (us * 1e-6) / 1e9 / peak,
                   "gate_up_us": ph["gate_up"], "down_us": ph["down"], "route_us": ph["route"],
                   "combine_us": ph["combine"],
                   "gate_up_frac": gu / (ph["gate_up"] * 1e-6) / 1e9 / peak
                   if ph["gate_up"] > 0 else None,
                   "down_frac": dn / (ph["down"] * 1e-6) / 1e9 / peak if ph["down"] > 0 else None,
                   "reps": len(times),
                   "l2": "weights larger than L2" if per_layer * n_layers > 4 * 129e6
                   else "layer fits in L2 (latency point)"}
            if n >= 256:
                fl = synth.algorithmic_flops(spec, n)
                rec["tflops"] = fl / (us * 1e-6) / 1e12
                rec["tensor_frac"] = rec["tflops"] / tflops_peak
                rec["tensor_peak_kind"] = tflops_kind
            if extra:
                rec["extra"] = "supplementary tensor-bound point (beyond the configs' token counts)"
            out.append(rec)
            if log:
                log(rec)
            del xs
        for lay in layers:
            lay.close()
        del layers
        torch.cuda.empty_cache()
    return out


def run_tier_points(dev, st, peak, spec, n, fractions=(1.0, 0.6, 0.3)):
    """Expert residency tiers: the decode workload with a fraction of the
    experts resident in device memory (chosen by the placement policy from
    the routing counts of 32 calibration batches) and the rest in pinned host
    memory behind the minimum slot pool (min(cold, n * top_k) slots).  Per
    fraction: time per forward, slot hit rate, and the bytes copied from host
    memory per call."""
    import torch
    from quantized_expert_ffn_warp_gb300 import moe
    w = synth.make_layer_device(spec, seed=200, device=dev)
    layer = moe.MoeLayer(spec, w, max_tokens=n)
    del w
    xs = [torch.from_numpy(synth.make_tokens(spec, n, seed=11, batch=b).view(np.float16)).to(dev)
          for b in range(16)]
    counts = np.zeros(spec.n_experts, np.int64)
    for b in range(32):
        x = torch.from_numpy(synth.make_tokens(spec, n, seed=12, batch=b).view(np.float16)).to(dev)
        counts += layer.route_topk(x, stream=st)["counts"].cpu().numpy()
    out = []
    try:
        for f in fractions:
            R = int(round(f * spec.n_experts))
            S = min(spec.n_experts - R, n * spec.top_k)
            layer.set_residency(moe.residency_plan(counts, R), S)
            s0 = layer.tier_stats()
            us, ph, touched, times = measure_layers([layer], xs, spec, n, st)
            s1 = layer.tier_stats()
            # forwards run: the sequence before capture, the warm-up period, the
            # timed repetitions and the eager profiling pass (16 steps each)
            forwards = 16 * (3 + len(times))
            hits, misses = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
            ab = synth.spec_algorithmic_bytes(spec, touched, n)
            out.append({"config": spec.name, "n": n, "resident_frac": f, "resident": R,
                        "slots": S, "us_per_forward": us, "tokens_per_s": n / (us * 1e-6),
                        "whole_layer_frac": ab / (us * 1e-6) / 1e9 / peak,
                        "slot_hit_rate": hits / max(hits + misses, 1),
                        "misses_per_call": misses / forwards,
                        "host_bytes_per_call": misses / forwards * synth.expert_bytes(spec),
                        "stage_us": ph["group"]})
    finally:
        layer.close()
    return out


def run_prenorm_cost(dev, st, spec, n):
    """What the RMSNorm in front costs inside a CUDA graph: the layer with the
    norm in front (moe_forward_prenorm on residual rows) against the plain
    layer on the very tokens the norm produces (same routing, same expert
    traffic), both timed as graph rotations over 4 layers and 16 batches."""
    import torch
    from quantized_expert_ffn_warp_gb300 import moe
    layers = [moe.MoeLayer(spec, synth.make_layer_device(spec, seed=300 + i, device=dev),
                           max_tokens=n) for i in range(4)]
    gain = torch.from_numpy(synth.make_norm_gain(spec).view(np.float16)).to(dev)
    resid = [torch.from_numpy(synth.make_residual(spec, n, seed=13, batch=b).view(np.float16))
             .to(dev) for b in range(16)]
    xn = [moe.rmsnorm(r, gain, NORM_EPS, stream=st) for r in resid]
    st.synchronize()
    try:
        us_plain, _, _, _ = measure_layers(layers, xn, spec, n, st)
        us_pre, _, _, _ = measure_layers(layers, resid, spec, n, st, prenorm_gain=gain)
        # the RMSNorm launch alone, in a graph of 16 calls
        g = torch.cuda.CUDAGraph()
        outs = [torch.empty_like(r) for r in resid]
        with torch.cuda.stream(st):
            for i in range(16):
                moe.rmsnorm(resid[i], gain, NORM_EPS, out=outs[i], stream=st)
            st.synchronize()
            with torch.cuda.graph(g, stream=st):
                for i in range(16):
                    moe.rmsnorm(resid[i], gain, NORM_EPS, out=outs[i], stream=st)
        def replay(k0, k):
            with torch.cuda.stream(st):
                for _ in range(k // 16):
                    g.replay()
        times, _ = timed_reps(replay, 0, 16, st, None, None, 20.0, 64)
        us_norm = 1e3 * statistics.median(times) / 16
    finally:
        for lay in layers:
            lay.close()
    return {"config": spec.name, "n": n, "us_forward_on_normalised_tokens": us_plain,
            "us_forward_prenorm": us_pre, "rmsnorm_cost_in_forward_us": us_pre - us_plain,
            "us_rmsnorm_alone": us_norm}


def cpu_config_points(seconds):
    """The oracle on 1 core and on all cores for the small and middle configs
    (bounded: at least one forward, up to `seconds` each)."""
    import oracle
    oracle.build()
    all_cores = oracle.num_threads()
    out = []
    for name, n in [("tiny", 4), ("e64_top2_zipf", 8), ("e256_top8_shared", 1),
                    ("e256_top8_shared", 16), ("e512_top4_shared", 1), ("e512_top4_shared", 4),
                    ("e512_top4_shared", 32), ("e512_top4_shared_2bit", 32)]:
        spec = synth.CONFIGS[name]
        layer = synth.make_layer(spec, 0)
        rec = {"config": name, "n": n}
        for cores in (1, all_cores):
            oracle.set_num_threads(cores)
            rate, calls, el, _ = cpu_oracle_rate(spec, n, seconds, layer)
            rec["tokens_per_s_%dcore%s" % (cores, "" if cores == 1 else "s")] = rate
        oracle.set_num_threads(all_cores)
        out.append(rec)
        del layer
    return out


def main():
    args = parse()
    spec = synth.CONFIGS[args.config]
    n = args.n or synth.TOKENS[args.config][-1 if args.config.startswith("e64_top2_sweep") else 0]
    if args.config.startswith("e64_top2_sweep") and args.n is None:
        n = 8
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, spec, n, rank, world)
        return

    import torch
    from quantized_expert_ffn_warp_gb300 import build as libbuild
    from quantized_expert_ffn_warp_gb300 import moe
    libbuild.build()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    dev = "cuda:%d" % local
    if args.quick:
        args.layers, args.batches = min(args.layers, 2), min(args.batches, 4)

    # layers (seeded per rank: independent replicas) and token batches
    layers, packed0 = [], None
    layer_seeds, token_seed = replica_seeds(rank, args.layers)
    for i in range(args.layers):
        packed = synth.make_layer(spec, seed=layer_seeds[i])
        if i == 0:
            packed0 = packed
        layers.append(moe.MoeLayer.from_packed(packed, max_tokens=max(n, 1), device=dev))
        if args.gemm_min_tokens is not None:
            layers[-1].set_gemm_min_tokens(args.gemm_min_tokens)
        if i:
            del packed
    gain = None
    if args.prenorm:   # inputs are residual rows; the layer sees their RMSNorm
        xs_np = [synth.make_residual(spec, n, seed=token_seed, batch=b)
                 for b in range(args.batches)]
        gain = torch.from_numpy(synth.make_norm_gain(spec).view(np.float16)).to(dev)
    else:
        xs_np = [synth.make_tokens(spec, n, seed=token_seed, batch=b) for b in range(args.batches)]
    xs = [torch.from_numpy(x.view(np.float16)).to(dev) for x in xs_np]
    outs = [torch.empty_like(xs[0]) for _ in range(args.batches)]
    st = torch.cuda.Stream(device=dev)
    info = layers[0].info()

    # touched experts per (layer, batch): from the library's own routing output
    touched = {}
    for li, L in enumerate(layers):
        for b, x in enumerate(xs):
            if args.prenorm:
                x = moe.rmsnorm(x, gain, NORM_EPS, stream=st)
            r = L.route_topk(x, stream=st)
            torch.cuda.synchronize()
            touched[(li, b)] = int((r["counts"] > 0).sum().item())

    def seq(i):
        return i % args.layers, i % args.batches

    def step(i, s):
        li, b = seq(i)
        if args.prenorm:
            layers[li].forward_prenorm(xs[b], gain, NORM_EPS, outs[b], stream=s)
        else:
            layers[li].forward(xs[b], outs[b], stream=s)

    # one rotation of (layer, batch) pairs; graphs of it and of its single steps
    period = int(np.lcm(args.layers, args.batches))
    runner = StepRunner(step, period, st, not args.no_graph)

    steps, warm = args.steps, max(args.warmup, 3)
    runner.run(0, warm)                   # exactly `warm` untimed steps
    st.synchronize()

    # timed: repetitions of exactly `steps` steps until >= 0.5 s and >= 128
    # forwards are timed; the median repetition gives the value
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    rep_ms, _ = timed_reps(runner.run, warm, steps, st, pg, dev, 500.0, 128)
    clocks = clk.stop()
    ms = statistics.median(rep_ms)
    value = job_rate(steps * n, world, ms)

    # per-kernel durations: the same sequence launched eagerly with events
    for L in layers:
        L.profile_enable(True)
    prof_steps = max(period, 64)
    with torch.cuda.stream(st):
        for i in range(prof_steps):
            step(i, st)
    st.synchronize()
    phase = {p: 0.0 for p in moe.PHASES}
    calls = 0
    for L in layers:
        d, c = L.profile_read()
        L.profile_enable(False)
        for p in d:
            phase[p] += d[p]
        calls += c
    phase_avg_us = {p: 1e3 * phase[p] / max(calls, 1) for p in phase}

    # algorithmic bytes of the gate/up kernel per launch (dominant kernel):
    # the touched experts' gate+up codes, scales and zeros (+ shared expert's)
    H = spec.hidden
    avg_touched = float(np.mean([touched[seq(i)] for i in range(prof_steps)]))
    gu_bytes = gate_up_bytes(spec, avg_touched, n)
    all_bytes = float(np.mean([synth.algorithmic_bytes(packed0, touched[seq(i)], n)
                               for i in range(prof_steps)]))
    peak, peak_kind = measured_peaks()
    gu_us = phase_avg_us["gate_up"]
    achieved = gu_bytes / (gu_us * 1e-6) / 1e9 if gu_us > 0 else None
    layer_us = 1e3 * ms / steps
    roofline = {
        "bound": "hbm", "kernel": "gate_up (dequant x MMA + SwiGLU)",
        "achieved": achieved, "peak": peak, "unit": "GB/s",
        "frac": achieved / peak if achieved else None, "peak_kind": peak_kind,
        "traffic": None if args.prenorm else recorded_traffic(args.config, n),
        "bytes_per_launch": gu_bytes, "us_per_launch": gu_us,
        "whole_layer": {"algorithmic_bytes": all_bytes, "us_per_call": layer_us,
                        "achieved_gbs": all_bytes / (layer_us * 1e-6) / 1e9,
                        "frac": all_bytes / (layer_us * 1e-6) / 1e9 / peak},
        "down": {"bytes_per_launch": down_bytes(spec, avg_touched),
                 "us_per_launch": phase_avg_us["down"],
                 "frac": down_bytes(spec, avg_touched) / (phase_avg_us["down"] * 1e-6) / 1e9 / peak
                 if phase_avg_us["down"] > 0 else None},
        "phase_us": phase_avg_us,
    }

    # end to end through the public API with pinned host buffers: the same
    # exact step count per repetition, host -> device and device -> host
    # copies of every step inside the timed region
    xh = [torch.from_numpy(x.view(np.float16)).pin_memory() for x in xs_np]
    oh = [torch.empty_like(x).pin_memory() for x in xh]

    def host_steps(k0, k):
        for i in range(k0, k0 + k):
            li, b = seq(i)
            moe.forward_host(layers[li], xh[b], oh[b], stream=st,
                             norm=(gain, NORM_EPS) if args.prenorm else None)
    t0 = time.perf_counter()
    e2e_ms, _ = timed_reps(host_steps, 0, steps, st, pg, dev, 300.0, 128)
    e2e = {"value": job_rate(steps * n, world, statistics.median(e2e_ms)), "unit": UNIT,
           "h2d_bytes_per_step": n * H * 2, "d2h_bytes_per_step": n * H * 2,
           "steps": steps, "repetitions": len(e2e_ms), "wall_s": time.perf_counter() - t0}

    for L in layers:
        L.close()
    layers = []
    torch.cuda.empty_cache()

    configs = tiers = prenorm_cost = None
    if rank == 0 and not args.quick and not args.no_configs:
        configs = run_config_points(dev, st, peak, CONFIG_POINTS)
        tiers = run_tier_points(dev, st, peak, spec, n)
        prenorm_cost = run_prenorm_cost(dev, st, spec, n)

    cpu = cpu_configs = None
    if rank == 0 and world == 1 and not args.no_cpu:
        rate, calls_c, el, cores = cpu_oracle_rate(spec, n, args.cpu_seconds, packed0,
                                                   prenorm=args.prenorm)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%d whole-layer forwards of %d tokens of layer instance 0 (%.1f s)"
                         % (calls_c, n, el)}
        if not args.quick and not args.no_configs:
            cpu_configs = cpu_config_points(2.0)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": ms / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "int%d-weights x f16 -> f32 accumulate" % spec.wbits,
            "data": "synthetic (seeded random layers and tokens)",
            "config": {"workload": workload_name(spec, n, args.prenorm), "n_tokens": n,
                       "gemm_min_tokens": info["gemm_min_tokens"] if args.gemm_min_tokens is None
                       else args.gemm_min_tokens,
                       "layers_rotated": args.layers, "batches_rotated": args.batches,
                       "cuda_graph": not args.no_graph,
                       "l2": "inputs larger than L2: each step streams a different layer "
                             "instance (%.0f MB of touched weights per call, %d instances of "
                             "%.2f GB)" % (all_bytes / 1e6, args.layers,
                                           info["weight_bytes"] / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "timing": {"repetitions": len(rep_ms), "steps_per_repetition": steps,
                       "median_ms": ms, "mean_ms": float(np.mean(rep_ms)),
                       "min_ms": float(np.min(rep_ms)), "max_ms": float(np.max(rep_ms)),
                       "timed_forwards": len(rep_ms) * steps},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            # kernels launched inside the timed regions (every repetition)
            "gpu_launches": kernels_per_forward(spec, n, info, args.prenorm) * steps * len(rep_ms),
            "gpu_launches_per_step": kernels_per_forward(spec, n, info, args.prenorm),
            "clocks": clocks,
            "touched_experts_avg": avg_touched,
            "configs": configs, "cpu_configs": cpu_configs, "residency": tiers,
            "prenorm_cost": prenorm_cost,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
