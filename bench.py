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
    ap.add_argument("--steps", type=int, default=200)
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
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
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
                 "--format=csv,noheader,nounits", "-lms", "200"],
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
    if rank != 0:
        return
    rate, calls, el, cores = cpu_oracle_rate(spec, n, args.cpu_seconds, prenorm=args.prenorm)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": calls, "warmup": 0, "ms_per_step": 1e3 * el / calls, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(spec, n, args.prenorm), "n_tokens": n},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d whole-layer forwards of %d tokens (%.1f s)" % (calls, n, el)},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


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

    # a graph holding one full rotation of (layer, batch) pairs
    period = int(np.lcm(args.layers, args.batches))
    graph = None
    if not args.no_graph:
        with torch.cuda.stream(st):
            for i in range(period):       # warm the exact sequence once
                step(i, st)
        st.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            with torch.cuda.graph(graph, stream=st):
                for i in range(period):
                    step(i, st)

    def run(k0, k):
        """k steps starting at step index k0 (graph replays cover whole periods)."""
        if graph is not None:
            assert k0 % period == 0 and k % period == 0
            for _ in range(k // period):
                graph.replay()
        else:
            for i in range(k0, k0 + k):
                step(i, st)

    steps = max(period, (args.steps // period) * period) if graph is not None else args.steps
    warm = max(args.warmup, 3)
    if graph is not None:
        warm = max(period, ((warm + period - 1) // period) * period)
    with torch.cuda.stream(st):
        run(0, warm)
    st.synchronize()

    def barrier():
        if pg:
            pg.barrier()

    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    with torch.cuda.stream(st):
        run(0, steps)
    e1.record(st)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier()
    clocks = clk.stop()
    ms = max_over_ranks(pg, e0.elapsed_time(e1), dev)
    value = job_rate(steps * n, world, ms)

    # per-kernel durations: the same sequence launched eagerly with events
    for L in layers:
        L.profile_enable(True)
    prof_steps = min(steps, max(period, 64))
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
    H, I, wb = spec.hidden, spec.inter, spec.wbits
    gu_expert = 2 * (I * H * wb // 8 + I * (H // 128) * 3)
    gu_shared = 2 * (spec.shared_inter * H * wb // 8 + spec.shared_inter * (H // 128) * 3) \
        if spec.has_shared else 0
    avg_touched = float(np.mean([touched[seq(i)] for i in range(prof_steps)]))
    gu_bytes = avg_touched * gu_expert + gu_shared + n * H * 2
    dn_expert = I * H * wb // 8 + H * (I // 128) * 3
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
        "down": {"bytes_per_launch": avg_touched * dn_expert + (
            spec.hidden * spec.shared_inter * wb // 8 + H * (spec.shared_inter // 128) * 3
            if spec.has_shared else 0), "us_per_launch": phase_avg_us["down"]},
        "phase_us": phase_avg_us,
    }

    # end to end through the public API with pinned host buffers
    xh = [torch.from_numpy(x.view(np.float16)).pin_memory() for x in xs_np]
    oh = [torch.empty_like(x).pin_memory() for x in xh]
    e2e_steps = min(steps, 100)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(st)
    for i in range(e2e_steps):
        li, b = seq(i)
        moe.forward_host(layers[li], xh[b], oh[b], stream=st,
                         norm=(gain, NORM_EPS) if args.prenorm else None)
    a1.record(st)
    a1.synchronize()
    e2e_ms = max_over_ranks(pg, a0.elapsed_time(a1), dev)
    e2e = {"value": job_rate(e2e_steps * n, world, e2e_ms), "unit": UNIT,
           "h2d_bytes_per_step": n * H * 2, "d2h_bytes_per_step": n * H * 2,
           "wall_s": time.perf_counter() - t0}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        for L in layers:
            L.close()
        layers = []
        torch.cuda.empty_cache()
        rate, calls_c, el, cores = cpu_oracle_rate(spec, n, args.cpu_seconds, packed0,
                                                   prenorm=args.prenorm)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%d whole-layer forwards of %d tokens of layer instance 0 (%.1f s)"
                         % (calls_c, n, el)}

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
                       "cuda_graph": graph is not None,
                       "l2": "inputs larger than L2: each step streams a different layer "
                             "instance (%.0f MB of touched weights per call, %d instances of "
                             "%.2f GB)" % (all_bytes / 1e6, args.layers,
                                           info["weight_bytes"] / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels_per_forward(spec, n, info, args.prenorm) * steps,
            "clocks": clocks,
            "touched_experts_avg": avg_touched,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
