#!/usr/bin/env python3
"""Throughput of one sparse-MoE FFN layer forward (route -> dispatch -> grouped SwiGLU -> combine)
on GB300, printed as one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one moe_layer_forward call over one batch of the workload (inputs resident in HBM).
Between timed steps a 256 MB buffer is written to flush L2. Each step is timed with CUDA events on
the launching stream; the K steps are bracketed by a barrier and a device synchronize.
`e2e` is the same metric through moe_layer_forward_host (pinned host x in, host out, copies in
the timed region), run as a serving loop runs it: calls rotate over three streams and three
workspaces, so the other calls' copies overlap one call's compute, and events bracket the whole
loop. The one-call-at-a-time latency is reported beside it as `e2e.serial`. `roofline` is for the
step's dominant kernel, timed live with events recorded between the layer's phases
(moe_layer_forward_profiled). `cpu_baseline` times the fp64 CPU
oracle on a bounded sample of the same workload. The headline workload is the largest one that
fits one GPU (the skewed prefill with a capacity limit); `per_config` times the fine-grained
prefill, the Gumbel prefill and the decode shape in the same run (device-resident inputs, L2
flushed between steps), each with its own layer and dominant-kernel rooflines.
With N > 1 (torchrun) every rank runs an independent replica of the layer (the layer has no
cross-token exchange): value = N*T / max time; `per_config` is then left out.
`--impl reference` times the oracle alone (rank 0; the other ranks exit) on the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (bf16, 1 GB300) and achieved fraction of roofline"
DEFAULT_CONFIG = "skewed_cap"  # the largest single-GPU workload: 11.75 GB of algorithmic bytes
# timed in the same run after the headline workload, each reported under "per_config"
PER_CONFIG = ("fine_grained", "gumbel", "decode")
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes per launch of the dominant kernels, from ncu captures of the current kernels (one
# line per workload and phase; see the file's header). Re-captured whenever a kernel changes.
NCU_DRAM_FILE = os.path.join(ROOT, "profiles", "ncu_dram_bytes.txt")


def read_ncu_dram(path=NCU_DRAM_FILE):
    """{(workload, phase): (scaling, read_bytes, write_bytes, captured_alg_bytes)} from the
    capture table."""
    out = {}
    if not os.path.exists(path):
        return out
    with open(path) as fh:
        for line in fh:
            f = line.split("#", 1)[0].split()
            if len(f) >= 5:
                out[(f[0], f[1])] = (f[2], float(f[3]), float(f[4]),
                                     float(f[5]) if len(f) > 5 else None)
    return out


def ncu_traffic(cfg, kernel, alg_bytes, table=None):
    """DRAM bytes (read + write) per launch of the dominant kernel from an ncu capture, or None.
    'launch' lines hold one full launch of the workload. 'alg' lines were captured on a smaller
    shape with the same rows per expert (the full launch exceeds a capture's size): their bytes
    are scaled by the ratio of the full launch's algorithmic bytes to the captured launch's."""
    t = read_ncu_dram() if table is None else table
    if (cfg.name, kernel) not in t:
        return None
    scaling, rd, wr, alg_cap = t[(cfg.name, kernel)]
    if scaling == "launch":
        return rd + wr
    if scaling == "alg" and alg_cap:
        return (rd + wr) * alg_bytes / alg_cap
    return None


def launches_per_step(cfg):
    """Kernels of one layer call with prepared weights: router (GEMM, selection, exact near-tie
    pass), dispatch (histogram with the scan and the tile list in its last CTA, scatter), gather,
    the two grouped GEMMs (or the two quantized FFN passes) and the combine; the overflow
    re-route adds its four kernels and a second dispatch."""
    n = 9
    if getattr(cfg, "reroute", False) and cfg.capacity_factor > 0:
        n += 4 + 2
    return n


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(prefix="moe_clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------------------ workload math
def touched_experts(counts, C):
    kept = [min(c, C) if C else c for c in counts]
    return sum(1 for c in kept if c > 0), sum(kept)


def weight_bytes_per_element(cfg):
    """HBM bytes per expert weight: 2 for bf16; bits/8 plus the fp16 scale and uint8 zero-point
    of each 128-weight group for quantized experts."""
    bits = getattr(cfg, "weight_bits", 0)
    return 2.0 if not bits else bits / 8.0 + 3.0 / 128.0


def layer_roofline(cfg, n_touched, n_kept, t_layer_s, peaks):
    P_tc = peaks["bf16_tflops"] * 1e12
    P_hbm = peaks["hbm_gbs"] * 1e9
    d, f, E, T, k, S = cfg.d, cfg.f, cfg.E, cfg.T, cfg.k, cfg.S
    F = 6.0 * T * k * d * f
    F_alg = 6.0 * n_kept * d * f + 6.0 * T * S * d * f + 2.0 * T * d * E
    B = (n_touched + S) * 3.0 * d * f * weight_bytes_per_element(cfg) + d * E * 2 + 2.0 * T * d * 2
    t_roof = max(F / P_tc, B / P_hbm)
    t_alg = max(F_alg / P_tc, B / P_hbm)
    return {"bound": "tensor" if F / P_tc >= B / P_hbm else "hbm",
            "F_flop": F, "F_alg_flop": F_alg, "B_bytes": B, "t_roof_us": t_roof * 1e6,
            "t_layer_us": t_layer_s * 1e6, "frac": t_roof / t_layer_s,
            "frac_alg": t_alg / t_layer_s}


def kernel_work(cfg, phase, n_touched, n_kept, n_tok_kept=None):
    """Algorithmic (flops, bytes) of one launch of a phase, from the config and the routing.
    n_tok_kept: tokens with at least one kept slot (all T when None)."""
    d, f, E, T, k, S = cfg.d, cfg.f, cfg.E, cfg.T, cfg.k, cfg.S
    rows = n_kept + S * T
    ne = n_touched + S
    wb = weight_bytes_per_element(cfg)
    if phase == "gate_up_gemm":
        return 4.0 * rows * d * f, ne * 2.0 * d * f * wb + rows * d * 2.0 + rows * f * 2.0
    if phase == "down_gemm":
        return 2.0 * rows * f * d, ne * 1.0 * f * d * wb + rows * f * 2.0 + rows * d * 2.0
    if phase == "router":
        return 2.0 * T * d * E, T * d * 2.0 + d * E * 2.0 + T * k * 8.0
    if phase == "combine":
        return 0.0, (n_kept + S * T) * d * 2.0 + T * d * 2.0 + T * k * 4.0
    if phase == "tiles_gather":
        # gathered rows written once; the x row of every token with a kept slot read once from
        # DRAM (repeat reads of a token's row hit L2; tokens whose slots were all dropped are
        # not read)
        n_tok = T if n_tok_kept is None else n_tok_kept
        return 0.0, n_kept * d * 2.0 + n_tok * d * 2.0
    if phase == "dispatch":
        return 0.0, T * k * 4.0 * 4
    return 0.0, 0.0


def roofline_for(phase, flops, nbytes, secs, peaks):
    """Tensor-bound when the launch's arithmetic intensity reaches the ridge, else HBM-bound."""
    if flops > 0:
        ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        if flops / max(nbytes, 1.0) >= ridge:
            ach = flops / secs / 1e12
            r = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                 "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"]}
            # beside the burst figure: the power-capped rate a seconds-long GEMM loop settles at
            if peaks.get("bf16_tflops_sustained"):
                r["frac_of_sustained"] = ach / peaks["bf16_tflops_sustained"]
            return r
    ach = nbytes / secs / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"]}


# ------------------------------------------------------------------------------ oracle timing
def oracle_sample_run(cfg, x_bits, Wg_bits, bias, u, get_expert, get_shared, n_tok, start=0):
    """Time the fp64 oracle on tokens [start, start + n_tok) taken as one batch."""
    import numpy as np
    import oracle as O
    sl = slice(start, start + n_tok)
    x64 = O.bf16_bits_to_f64(x_bits[sl])
    Wg64 = O.bf16_bits_to_f64(Wg_bits)
    uu = u[sl] if u is not None else None
    t0 = time.perf_counter()
    O.layer(x64, Wg64, cfg.k, get_expert, cfg.E, cfg.mode, bias, uu, cfg.tau,
            cfg.capacity_factor, n_shared=cfg.S, get_shared=get_shared,
            n_groups=cfg.n_groups, topk_groups=cfg.topk_groups, reroute=cfg.reroute)
    return time.perf_counter() - t0


class WidenedExperts:
    """bf16 expert weights (host numpy) widened to float64 on first use and kept; with bits > 0
    the oracle's own quantize-dequantize of them (model load, outside any timing)."""

    def __init__(self, Wg, Wu, Wd, bits=0):
        self.src = (Wg, Wu, Wd)
        self.bits = bits
        self.cache = {}

    def __call__(self, e):
        import oracle as O
        if e not in self.cache:
            ws = tuple(O.bf16_bits_to_f64(w[e]) for w in self.src)
            if self.bits:
                ws = tuple(O.dequantize_groupwise(*O.quantize_groupwise(w, self.bits))
                           for w in ws)
            self.cache[e] = ws
        return self.cache[e]


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def routing_inputs_np(inp):
    import workloads as W
    x_bits = W.bf16_bits(inp["x"])
    Wg_bits = W.bf16_bits(inp["W_g"])
    bias = inp["bias"].double().cpu().numpy()
    u = inp["u"].cpu().numpy() if inp.get("u") is not None else None
    return x_bits, Wg_bits, bias, u


def host_weights_np(inp, bits=0):
    import workloads as W
    ex = WidenedExperts(W.bf16_bits(inp["W_gate"]), W.bf16_bits(inp["W_up"]),
                        W.bf16_bits(inp["W_down"]), bits)
    sh = None
    if inp.get("Ws_gate") is not None:
        sh = WidenedExperts(W.bf16_bits(inp["Ws_gate"]), W.bf16_bits(inp["Ws_up"]),
                            W.bf16_bits(inp["Ws_down"]), bits)
    return ex, sh


def cpu_baseline(cfg, inp, target_s=12.0):
    """The oracle as it stands, timed on a bounded sample: the first n tokens taken as one
    batch (n = T when a whole batch fits the time budget, then repeated while under it)."""
    x_bits, Wg_bits, bias, u = routing_inputs_np(inp)
    ex, sh = host_weights_np(inp, cfg.weight_bits)
    n0 = min(32, cfg.T)
    oracle_sample_run(cfg, x_bits, Wg_bits, bias, u, ex, sh, n0)       # widen + warm
    t0 = oracle_sample_run(cfg, x_bits, Wg_bits, bias, u, ex, sh, n0)
    per_tok = max(t0 / n0, 1e-7)
    n = int(max(n0, min(cfg.T, 0.5 * target_s / per_tok)))
    if n < cfg.T:
        for e in range(cfg.E):   # widen every expert the larger sample may hit (model load)
            ex(e)
    total_t, runs = 0.0, 0
    while runs == 0 or (total_t < target_s and runs < 50):
        total_t += oracle_sample_run(cfg, x_bits, Wg_bits, bias, u, ex, sh, n)
        runs += 1
    return {"value": n * runs / total_t, "unit": "tokens/s", "cores": cpu_cores(),
            "kind": "oracle",
            "sample": f"tokens 0..{n - 1} of the workload as one batch ({n} of {cfg.T}), "
                      f"{runs} run(s), {total_t:.1f} s; float64 numpy oracle, expert weights "
                      f"widened once beforehand",
            "seconds": total_t}


# ------------------------------------------------------------------------------ reference arm
def run_reference(args, cfg):
    import numpy as np
    import workloads as W
    inp = W.make_inputs(cfg, weights_device="cpu")
    x_bits, Wg_bits, bias, u = routing_inputs_np(inp)
    ex, sh = host_weights_np(inp, cfg.weight_bits)
    budget = 150.0
    n0 = min(8, cfg.T)
    oracle_sample_run(cfg, x_bits, Wg_bits, bias, u, ex, sh, n0)          # widen + warm
    for e in range(cfg.E):
        ex(e)
    t0 = oracle_sample_run(cfg, x_bits, Wg_bits, bias, u, ex, sh, n0)
    per_tok = max(t0 / n0, 1e-6)
    n = int(max(1, min(cfg.T, budget / (args.steps + args.warmup) / per_tok)))
    times = []
    for i in range(args.warmup + args.steps):
        start = (i * n) % max(1, cfg.T - n + 1)
        t = oracle_sample_run(cfg, x_bits, Wg_bits, bias, u, ex, sh, n, start)
        if i >= args.warmup:
            times.append(t)
    mean = sum(times) / len(times)
    value = n / mean
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": config_dict(cfg),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle",
                             "cores": cpu_cores(),
                             "sample": f"{n} consecutive tokens per step as one batch "
                                       f"(window moves each step); float64 numpy oracle"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(cfg):
    return {"workload": cfg.name + ": " + cfg.description, "T": cfg.T, "d": cfg.d, "E": cfg.E,
            "n_shared": cfg.S, "top_k": cfg.k, "d_ff": cfg.f, "mode": cfg.mode, "tau": cfg.tau,
            "capacity_factor": cfg.capacity_factor, "seed": cfg.seed,
            "n_groups": cfg.n_groups, "topk_groups": cfg.topk_groups,
            "overflow_reroute": cfg.reroute, "weight_bits": cfg.weight_bits,
            "l2": "flushed between timed steps (256 MB write)", "parallelism": "replicas"}


# ------------------------------------------------------------------------------ our arm
def load_workload(M, W, cfg, dev):
    """The workload's seeded inputs on the device and the one-time weight preparation (outside
    any timed region): the router weights' transpose, and the fp16 re-encoding of W_down or the
    group-wise quantization of every expert matrix. Returns (inp_host, inp, weights, keep,
    pack_ms); `keep` holds the prepared tensors the weights struct points at."""
    import torch
    inp_host = W.make_inputs(cfg, weights_device=dev)
    inp = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp_host.items()}
    pk0, pk1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pk0.record()
    keep = {"W_g_t": M.prepare_router(inp["W_g"])}
    if cfg.weight_bits:
        names = ("W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down")
        keep["q"] = {n: (M.quantize_weights(inp[n], cfg.weight_bits) if inp.get(n) is not None
                         else None) for n in names}
        keep["qstruct"] = M.make_qweights(*[keep["q"][n] for n in names])
    else:
        keep["Wd16"] = M.packed_f16(inp["W_down"])
        keep["Wsd16"] = (M.packed_f16(inp["Ws_down"]) if inp.get("Ws_down") is not None
                         else None)
    pk1.record()
    torch.cuda.synchronize()
    if cfg.weight_bits:
        weights = M.make_weights(inp["W_g"], inp["bias"], None, None, None,
                                 quant=keep["qstruct"], W_g_t=keep["W_g_t"])
    else:
        weights = M.make_weights(inp["W_g"], inp["bias"], inp["W_gate"], inp["W_up"],
                                 inp["W_down"], inp.get("Ws_gate"), inp.get("Ws_up"),
                                 inp.get("Ws_down"), keep["Wd16"], keep["Wsd16"],
                                 W_g_t=keep["W_g_t"])
    return inp_host, inp, weights, keep, pk0.elapsed_time(pk1)


def timed_steps(step, flush, stream, n):
    """Per-step ms of n calls of step(), each bracketed by CUDA events on the launching stream,
    with L2 flushed before each."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def phase_times(M, mc, weights, inp, out, ro, ws, flush, n):
    """Median ms of each phase of n layer calls through moe_layer_forward_profiled (the same
    kernels with events recorded between the phases); medians, so a host stall that lets the
    queue drain inflates one call's phase and not the figure."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(n)]
    for i in range(n):
        flush.fill_(i & 0xFF)
        M.layer_forward_profiled(mc, weights, inp["x"], inp.get("u"), out, ro, ws, evs[i])
    torch.cuda.synchronize()
    return {ph: statistics.median(e[j].elapsed_time(e[j + 1]) for e in evs)
            for j, ph in enumerate(M.PROFILE_PHASES)}


def tokens_with_kept_slot(slot_pos, T, k):
    """Tokens at least one of whose k slots was kept (slot_pos >= 0)."""
    return int((slot_pos.view(T, k) >= 0).any(dim=1).sum().item())


def workload_report(cfg, ms, phase_ms, counts_h, peaks, peak_src, n_tok_kept=None):
    """Layer roofline, the dominant kernel's roofline, per-phase fractions and routing figures."""
    C = M_capacity(cfg)
    n_touched, n_kept = touched_experts(counts_h, C)
    lr = layer_roofline(cfg, n_touched, n_kept, ms / 1e3, peaks)
    dom = max(phase_ms, key=phase_ms.get)
    fl, by = kernel_work(cfg, dom, n_touched, n_kept, n_tok_kept)
    roof = roofline_for(dom, fl, by, phase_ms[dom] / 1e3, peaks)
    roof["kernel"] = dom
    roof["traffic"] = ncu_traffic(cfg, dom, by)
    roof["peak_source"] = f"{peak_src} ({'bf16 burst' if roof['unit'] == 'TFLOP/s' else 'copy'})"
    kernels = {}
    for ph, t in phase_ms.items():
        f_, b_ = kernel_work(cfg, ph, n_touched, n_kept, n_tok_kept)
        r = roofline_for(ph, f_, b_, t / 1e3, peaks) if t > 0 else {}
        kernels[ph] = {"us": t * 1e3, **{kk: r[kk] for kk in ("bound", "frac", "frac_of_sustained")
                                         if kk in r}}
    routing = {"experts_hit": n_touched, "kept_slots": n_kept, "tokens_kept": n_tok_kept,
               "capacity": C,
               "dropped_slots": cfg.T * cfg.k - n_kept, "max_load": max(counts_h),
               "mean_load": cfg.T * cfg.k / cfg.E}
    return lr, roof, kernels, routing


def measure_other(M, W, name, dev, steps, warmup, peaks, peak_src, local):
    """One more workload timed in the same process (device-resident inputs, L2 flushed between
    steps, CUDA events): tokens/s, latency, layer and dominant-kernel rooflines, clocks."""
    import torch
    cfg = W.CONFIGS[name]
    _, inp, weights, keep, _ = load_workload(M, W, cfg, dev)
    mc = M.MoeConfig.from_layer(cfg)
    ws = M.alloc_workspace(mc, dev)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    slot_pos = torch.empty(cfg.T * cfg.k, dtype=torch.int32, device=dev)
    ro = M.make_route_out(counts=counts, slot_pos=slot_pos)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        M.layer_forward(mc, weights, inp["x"], inp.get("u"), out, ro, ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    step_ms = timed_steps(step, flush, stream, steps)
    clk = clocks.stop()
    phase_ms = phase_times(M, mc, weights, inp, out, ro, ws, flush, steps)
    faults = M.device_status(ws)
    if faults:
        raise SystemExit(f"device fault bits {faults:#x} in workload {name}")
    ms = sum(step_ms) / len(step_ms)
    lr, roof, kernels, routing = workload_report(cfg, ms, phase_ms, counts.cpu().tolist(), peaks,
                                                 peak_src,
                                                 tokens_with_kept_slot(slot_pos, cfg.T, cfg.k))
    del inp, weights, keep, ws, flush
    return {"workload": cfg.name + ": " + cfg.description, "value": cfg.T / (ms / 1e3),
            "unit": "tokens/s", "ms_per_step": ms, "ms_per_step_median": statistics.median(step_ms),
            "steps": steps, "warmup": warmup, "layer_roofline": lr, "roofline": roof,
            "kernels": kernels, "routing": routing, "clocks": clk,
            "gpu_launches": launches_per_step(cfg) * steps}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the --config workload (no per_config object)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import workloads as W
    cfg = W.CONFIGS[args.config]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, cfg)
        return

    import torch
    import sparse_moe_layer_route_gb300 as M
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    peaks, peak_src = load_peaks()

    dev = f"cuda:{local}"
    inp_host, inp, weights, keep, pack_ms = load_workload(M, W, cfg, dev)
    mc = M.MoeConfig.from_layer(cfg)
    ws = M.alloc_workspace(mc, dev)
    T, k, E, d = cfg.T, cfg.k, cfg.E, cfg.d
    out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    slot_pos = torch.empty(T * k, dtype=torch.int32, device=dev)
    ro = M.make_route_out(counts=counts, slot_pos=slot_pos)
    u = inp.get("u")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()

    def step():
        M.layer_forward(mc, weights, inp["x"], u, out, ro, ws)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    faults = M.device_status(ws)
    if faults:
        raise SystemExit(f"device fault bits {faults:#x} during warm-up")

    # ---- timed region: K steps, L2 flushed between them
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    ms_median = statistics.median(step_ms)

    # ---- phase breakdown through the profiled entry point (same kernels, events in between)
    phase_ms = phase_times(M, mc, weights, inp, out, ro, ws, flush, min(args.steps, 200))

    # ---- the same step replayed from a CUDA graph (launch overhead removed; L2 still flushed)
    graph = graph_replay(step, flush, stream, min(args.steps, 200))

    # ---- e2e: host buffers through moe_layer_forward_host (pinned x in, out back to the host,
    # both copies inside every call). Two measurements:
    #  * serial: one call at a time, L2 flushed before each, CUDA events around each call (latency);
    #  * serving loop (the reported value): successive calls rotate over three streams and three
    #    workspaces, as a server buffers its batches, so the other calls' copies run on the copy
    #    engines while one call computes (a stream runs its copy-in, compute and copy-out in order,
    #    so three keep the compute busy when the copies take up to its time each); events bracket the whole loop, so every step's
    #    copies and compute are inside the timed region. It is used when the expert weights one
    #    step streams are more than twice the L2 flush size (no flush needed); otherwise the
    #    serial figure is reported. The same loop on device buffers is reported beside it.
    x_h = inp_host["x"].pin_memory()
    u_h = inp_host["u"].pin_memory() if inp_host.get("u") is not None else None
    NBUF = 3
    out_h = [torch.empty((T, d), dtype=torch.bfloat16).pin_memory() for _ in range(NBUF)]
    ws2 = [ws] + [M.alloc_workspace(mc, dev) for _ in range(NBUF - 1)]
    # non-default streams only: work on the legacy default stream would order itself against
    # the other streams' copies
    streams2 = [torch.cuda.Stream(device=dev) for _ in range(NBUF)]
    n_e2e = min(args.steps, 200)
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    for i in range(3):
        M.layer_forward_host(mc, weights, x_h, u_h, out_h[0], ws)
    torch.cuda.synchronize()
    for i in range(n_e2e):
        flush.fill_(i & 0xFF)
        e_s[i].record(stream)
        M.layer_forward_host(mc, weights, x_h, u_h, out_h[0], ws)
        e_e[i].record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = sum(a.elapsed_time(b) for a, b in zip(e_s, e_e)) / n_e2e
    n_touched_now = touched_experts(counts.cpu().tolist(), M_capacity(cfg))[0]
    streamed = (n_touched_now + cfg.S) * 3 * cfg.d * cfg.f * weight_bytes_per_element(cfg)
    flush_each = streamed < 2 * L2_FLUSH_BYTES
    for i in range(2 * NBUF):
        M.layer_forward_host(mc, weights, x_h, u_h, out_h[i % NBUF], ws2[i % NBUF],
                             stream=streams2[i % NBUF])
    torch.cuda.synchronize()
    out_d2 = [out] + [torch.empty_like(out) for _ in range(NBUF - 1)]
    ro2 = [ro] + [M.make_route_out() for _ in range(NBUF - 1)]

    def serving_loop(host):
        """Per-step ms of n_e2e calls rotating over the streams and workspaces."""
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for st_b in streams2:
            st_b.wait_event(p0)
        for i in range(n_e2e):
            j = i % NBUF
            if host:
                M.layer_forward_host(mc, weights, x_h, u_h, out_h[j], ws2[j], stream=streams2[j])
            else:
                M.layer_forward(mc, weights, inp["x"], u, out_d2[j], ro2[j], ws2[j],
                                stream=streams2[j])
        for st_b in streams2:
            stream.wait_stream(st_b)
        p1.record(stream)
        torch.cuda.synchronize()
        return p0.elapsed_time(p1) / n_e2e

    # with weights that fit L2 a flush would have to sit inside the loop: report the serial figure
    if not flush_each:  # one untimed pass of each loop first
        serving_loop(True)
        serving_loop(False)
    loop_ms = serving_loop(True) if not flush_each else None
    loop_dev_ms = serving_loop(False) if not flush_each else None
    e2e_ms = loop_ms if loop_ms is not None else e2e_serial_ms
    clk = clocks.stop()
    faults = 0
    for w_ in ws2:
        faults |= M.device_status(w_)
    if faults:
        raise SystemExit(f"device fault bits {faults:#x} during the timed region")
    h2d = T * d * 2 + (T * E * 4 if u_h is not None else 0)
    d2h = T * d * 2

    # ---- max over ranks (replicas: no data-path collective, only this timing reduction)
    ms, e2e_ms, e2e_serial_ms = max_over_ranks([ms, e2e_ms, e2e_serial_ms], dist, dev)
    if loop_dev_ms is not None:
        loop_dev_ms = max_over_ranks([loop_dev_ms], dist, dev)[0]

    lr, roof, kernels, routing = workload_report(cfg, ms, phase_ms, counts.cpu().tolist(), peaks,
                                                 peak_src, tokens_with_kept_slot(slot_pos, T, k))
    # ---- the oracle on the host cores, on a bounded sample of the same workload
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, inp_host_weights(inp_host, inp))
    # ---- the other workloads, timed in the same run (one GPU only; the scaling runs skip them)
    per_config = None
    if world == 1 and not args.no_per_config:
        del inp, weights, keep, ws, ws2, flush, x_h, u_h, out_h, out_d2
        torch.cuda.empty_cache()
        per_config = {}
        for name in PER_CONFIG:
            if name != cfg.name:
                per_config[name] = measure_other(M, W, name, dev, min(args.steps, 100),
                                                 args.warmup, peaks, peak_src, local)
                torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {"metric": METRIC, "value": replica_throughput(world, T, ms), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": (f"int{cfg.weight_bits} weights x fp16 activations, fp32 accumulate"
                      if cfg.weight_bits else "bf16"),
            "data": "synthetic (seeded inputs, random-init weights)",
            "config": config_dict(cfg),
            "roofline": roof,
            "layer_roofline": lr,
            "kernels": kernels,
            "e2e": {"value": replica_throughput(world, T, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "mode": ("serving loop: calls rotate over 3 streams and 3 workspaces; "
                             "events around the whole loop; L2 not flushed: each step streams "
                             "%.2f GB of expert weights" % (streamed / 1e9)
                             if loop_ms is not None else
                             "serial: one call at a time, L2 flushed before each, events around "
                             "each call (the weights fit L2, so a loop would need the flush "
                             "inside its window)"),
                    "serial": {"value": replica_throughput(world, T, e2e_serial_ms),
                               "ms_per_step": e2e_serial_ms,
                               "mode": "one call at a time, L2 flushed before each, events around "
                                       "each call"},
                    "device_serving_loop": (None if loop_dev_ms is None else
                                            {"value": replica_throughput(world, T, loop_dev_ms),
                                             "ms_per_step": loop_dev_ms,
                                             "mode": "the same loop through moe_layer_forward "
                                                     "on device buffers (no copies)"})},
            "gpu_launches": launches_per_step(cfg) * args.steps,
            "clocks": clk,
            "routing": routing,
            "ms_per_step_median": ms_median,
            "graph_replay": graph,
            "weight_pack_ms": pack_ms,
            "wall_s_timed": wall,
            "per_config": per_config}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def graph_replay(step, flush, stream, n):
    """Median per-step time of `step` captured once in a CUDA graph and replayed n times, with the
    L2 flushed between replays (outside the graph)."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        st = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            flush.fill_(i & 0xFF)
            st[i].record(stream)
            g.replay()
            en[i].record(stream)
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in zip(st, en))
        return {"ms_per_step_median": ms, "steps": n}
    except RuntimeError as exc:  # a capture the driver refuses is reported, not fatal
        return {"error": str(exc).splitlines()[0][:200]}


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings over the process group (identity for one process)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    import torch
    tt = torch.tensor(values, device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return tt.tolist()


def replica_throughput(world, tokens_per_replica, ms):
    """Whole-job tokens/s when every rank runs one replica in `ms` milliseconds (max over ranks)."""
    return world * tokens_per_replica / (ms / 1e3)


def M_capacity(cfg):
    """Capacity of the config, as the library computes it (None: no limit)."""
    if cfg.capacity_factor <= 0:
        return None
    from fractions import Fraction
    import numpy as np
    return math.ceil(Fraction(float(np.float32(cfg.capacity_factor))) * cfg.T * cfg.k / cfg.E)


def inp_host_weights(inp_host, inp_dev):
    """Routing inputs from the host copy; expert weights copied from the device."""
    out = dict(inp_host)
    for key in ("W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down"):
        if inp_dev.get(key) is not None:
            out[key] = inp_dev[key].cpu()
    return out


if __name__ == "__main__":
    main()
