"""Seeded synthetic inputs for the sparse-MoE layer, shared by the CUDA path's tests/bench and the
CPU oracle.

This module only draws random numbers and rounds them to the layer's storage types. It holds
none of the layer's arithmetic (no routing, no top-k, no FFN), so neither side can inherit a
mistake from the other through it.

Draw recipe (fixed order, so every tensor is reproducible from the config's seed):
  * a CPU torch.Generator seeded with `seed` draws, in this order,
      x      [T, d]  ~ N(0, 1)           -> bf16 (round to nearest even)
      W_g    [d, E]  ~ N(0, 1/d)         -> bf16
      bias   [E]     fp32, per the config's bias recipe
      u      [T, E]  fp32 ~ U(0, 1), clamped to >= 2^-24 (GUMBEL configs only)
  * a generator on the weights' device seeded with `seed + 1000` draws, expert by expert,
      W_gate [E, d, f] ~ N(0, 1/d), W_up [E, d, f] ~ N(0, 1/d), W_down [E, f, d] ~ N(0, 1/f)
    then the shared experts' W_gate/W_up/W_down in the same way, all rounded to bf16.
  "N(0, v)" names the variance, so std = sqrt(v).

The expert weights of the large layers are ~11 GB, so they are drawn on the GPU when one is
present; the routing inputs are drawn on the CPU so that their bytes do not depend on the GPU.
"""
from __future__ import annotations

import hashlib
import json
import math
import os
from dataclasses import dataclass, field, asdict

import torch

PLAIN, BIAS_SELECT, GUMBEL = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    f: int
    S: int = 0                 # shared experts
    mode: int = PLAIN
    tau: float = 1.0
    capacity_factor: float = 0.0   # <= 0: no capacity limit
    seed: int = 0
    bias: str = "zero"         # "zero" | "normal" | "zipf"
    bias_var: float = 0.0
    zipf_s: float = 1.1
    n_groups: int = 0          # group-limited routing (0: off)
    topk_groups: int = 0
    reroute: bool = False      # Level-2 overflow re-route (with a capacity limit)
    weight_bits: int = 0       # 0: bf16 experts; 4 / 8: group-wise quantized experts
    description: str = ""

    def as_dict(self):
        return asdict(self)


CONFIGS = {
    "tiny": LayerConfig(
        "tiny", T=128, d=256, E=8, k=2, f=512, S=0, mode=PLAIN, seed=0,
        description="tiny layer: T=128 d=256 E=8 k=2 d_ff=512, plain top-2"),
    "fine_grained": LayerConfig(
        "fine_grained", T=4096, d=2048, E=64, k=6, f=1408, S=2, mode=BIAS_SELECT, seed=1,
        bias="normal", bias_var=0.1,
        description="fine-grained prefill: T=4096 d=2048 E=64+2 shared k=6 d_ff=1408, "
                    "bias-adjusted selection"),
    "decode": LayerConfig(
        "decode", T=64, d=7168, E=128, k=2, f=2048, S=1, mode=PLAIN, seed=2,
        description="decode shape: T=64 d=7168 E=128+1 shared k=2 d_ff=2048"),
    "skewed_cap": LayerConfig(
        "skewed_cap", T=16384, d=7168, E=128, k=2, f=2048, S=0, mode=BIAS_SELECT,
        capacity_factor=1.25, seed=3, bias="zipf", zipf_s=1.1,
        description="skewed prefill: T=16384 d=7168 E=128 k=2 d_ff=2048, Zipf(1.1) bias, "
                    "capacity ceil(1.25*T*k/E)"),
    "skewed_cap_reroute": LayerConfig(
        "skewed_cap_reroute", T=16384, d=7168, E=128, k=2, f=2048, S=0, mode=BIAS_SELECT,
        capacity_factor=1.25, seed=3, bias="zipf", zipf_s=1.1, reroute=True,
        description="the skewed prefill with Level-2 overflow re-route: dropped slots move to "
                    "the best expert with room"),
    "decode_int8": LayerConfig(
        "decode_int8", T=64, d=7168, E=128, k=2, f=2048, S=1, mode=PLAIN, seed=2, weight_bits=8,
        description="the decode shape with 8-bit group-wise quantized experts (128 weights per "
                    "group)"),
    "decode_int4": LayerConfig(
        "decode_int4", T=64, d=7168, E=128, k=2, f=2048, S=1, mode=PLAIN, seed=2, weight_bits=4,
        description="the decode shape with 4-bit group-wise quantized experts (128 weights per "
                    "group)"),
    # profiling size of the skewed prefill with re-route: the same routing (x, W_g and the bias
    # are drawn before the experts), d_ff = 128 (about 1 GB on the device)
    "skewed_reroute_f128": LayerConfig(
        "skewed_reroute_f128", T=16384, d=7168, E=128, k=2, f=128, S=0, mode=BIAS_SELECT,
        capacity_factor=1.25, seed=3, bias="zipf", zipf_s=1.1, reroute=True,
        description="the skewed prefill with re-route at d_ff=128 (profiling size)"),
    # profiling size of the skewed prefill's router and dispatch: the same routing without the
    # re-route, d_ff = 128 (about 2.5 GB on the device with the workspace)
    "skewed_f128": LayerConfig(
        "skewed_f128", T=16384, d=7168, E=128, k=2, f=128, S=0, mode=BIAS_SELECT,
        capacity_factor=1.25, seed=3, bias="zipf", zipf_s=1.1,
        description="the skewed prefill at d_ff=128 (profiling size of its router)"),
    # profiling size of the decode shape (32 routed experts: about 3 GB of weights on the device)
    "decode_e32": LayerConfig(
        "decode_e32", T=64, d=7168, E=32, k=2, f=2048, S=1, mode=PLAIN, seed=2,
        description="decode shape with 32 routed experts + 1 shared, bf16 experts (profiling "
                    "size)"),
    "decode_e32_int4": LayerConfig(
        "decode_e32_int4", T=64, d=7168, E=32, k=2, f=2048, S=1, mode=PLAIN, seed=2,
        weight_bits=4,
        description="decode shape with 32 routed experts + 1 shared, 4-bit experts (profiling "
                    "size)"),
    "decode_e32_int8": LayerConfig(
        "decode_e32_int8", T=64, d=7168, E=32, k=2, f=2048, S=1, mode=PLAIN, seed=2,
        weight_bits=8,
        description="decode shape with 32 routed experts + 1 shared, 8-bit experts (profiling "
                    "size)"),
    "gumbel": LayerConfig(
        "gumbel", T=8192, d=4096, E=16, k=2, f=14336, S=0, mode=GUMBEL, tau=0.5, seed=4,
        description="Gumbel top-2: T=8192 d=4096 E=16 k=2 d_ff=14336, tau=0.5"),
    # profiling sizes of the two prefill shapes: the same rows per expert (gumbel: T k / E =
    # 1024; skewed: mean 256 with capacity 320) at about 1.4 GB of expert weights each
    "gumbel_e4": LayerConfig(
        "gumbel_e4", T=2048, d=4096, E=4, k=2, f=14336, S=0, mode=GUMBEL, tau=0.5, seed=4,
        description="Gumbel top-2 with 4 experts: T=2048 d=4096 k=2 d_ff=14336 (profiling "
                    "size)"),
    "skewed_e16": LayerConfig(
        "skewed_e16", T=2048, d=7168, E=16, k=2, f=2048, S=0, mode=BIAS_SELECT,
        capacity_factor=1.25, seed=3, bias="zipf", zipf_s=1.1,
        description="skewed prefill with 16 experts: T=2048 d=7168 k=2 d_ff=2048, Zipf(1.1) "
                    "bias, capacity ceil(1.25*T*k/E) = 320 (profiling size)"),
}


def small_config(name="small", T=64, d=128, E=8, k=2, f=128, S=0, mode=PLAIN, tau=1.0,
                 capacity_factor=0.0, seed=0, bias="zero", bias_var=0.0, zipf_s=1.1,
                 n_groups=0, topk_groups=0, reroute=False, weight_bits=0):
    """A config for tests at sizes the oracle finishes in seconds."""
    return LayerConfig(name, T=T, d=d, E=E, k=k, f=f, S=S, mode=mode, tau=tau,
                       capacity_factor=capacity_factor, seed=seed, bias=bias,
                       bias_var=bias_var, zipf_s=zipf_s, n_groups=n_groups,
                       topk_groups=topk_groups, reroute=reroute, weight_bits=weight_bits)


def skew_scale() -> float:
    """Scale c of the Zipf bias, written by oracle/calibrate_skew.py."""
    with open(os.path.join(_HERE, "skew_calibration.json")) as fh:
        return float(json.load(fh)["c"])


def zipf_log_pmf(E: int, s: float) -> torch.Tensor:
    """ln p_r for p_r proportional to r^-s, r = 1..E (float64)."""
    r = torch.arange(1, E + 1, dtype=torch.float64)
    logw = -s * torch.log(r)
    return logw - torch.logsumexp(logw, 0)


def _sha(t: torch.Tensor) -> str:
    return hashlib.sha256(t.detach().cpu().contiguous().view(torch.uint8).numpy().tobytes()
                          ).hexdigest()


def make_routing_inputs(cfg: LayerConfig, zipf_scale: float | None = None):
    """x, W_g, bias, u on the CPU (see the module docstring for the recipe)."""
    g = torch.Generator(device="cpu").manual_seed(cfg.seed)
    x = torch.randn(cfg.T, cfg.d, generator=g).to(torch.bfloat16)
    W_g = (torch.randn(cfg.d, cfg.E, generator=g) * math.sqrt(1.0 / cfg.d)).to(torch.bfloat16)
    if cfg.bias == "zero":
        bias = torch.zeros(cfg.E, dtype=torch.float32)
    elif cfg.bias == "normal":
        bias = (torch.randn(cfg.E, generator=g) * math.sqrt(cfg.bias_var)).to(torch.float32)
    elif cfg.bias == "zipf":
        perm = torch.randperm(cfg.E, generator=g)          # expert e gets Zipf rank perm[e]+1
        c = skew_scale() if zipf_scale is None else zipf_scale
        bias = (c * zipf_log_pmf(cfg.E, cfg.zipf_s)[perm]).to(torch.float32)
    else:
        raise ValueError(cfg.bias)
    u = None
    if cfg.mode == GUMBEL:
        u = torch.rand(cfg.T, cfg.E, generator=g).clamp_(min=2.0 ** -24)
    return {"x": x, "W_g": W_g, "bias": bias, "u": u}


def make_expert_weights(cfg: LayerConfig, device="cpu"):
    """Routed and shared expert weights, drawn expert by expert on `device` (bf16)."""
    g = torch.Generator(device=device).manual_seed(cfg.seed + 1000)
    sd, sf = math.sqrt(1.0 / cfg.d), math.sqrt(1.0 / cfg.f)

    def stack(n, rows, cols, std):
        out = torch.empty(n, rows, cols, dtype=torch.bfloat16, device=device)
        for e in range(n):
            out[e] = (torch.randn(rows, cols, generator=g, device=device) * std).to(torch.bfloat16)
        return out

    W_gate = stack(cfg.E, cfg.d, cfg.f, sd)
    W_up = stack(cfg.E, cfg.d, cfg.f, sd)
    W_down = stack(cfg.E, cfg.f, cfg.d, sf)
    if cfg.S > 0:
        Ws_gate = stack(cfg.S, cfg.d, cfg.f, sd)
        Ws_up = stack(cfg.S, cfg.d, cfg.f, sd)
        Ws_down = stack(cfg.S, cfg.f, cfg.d, sf)
    else:
        Ws_gate = Ws_up = Ws_down = None
    return {"W_gate": W_gate, "W_up": W_up, "W_down": W_down,
            "Ws_gate": Ws_gate, "Ws_up": Ws_up, "Ws_down": Ws_down}


def make_inputs(cfg: LayerConfig, weights_device="cpu", zipf_scale: float | None = None):
    """All inputs of one layer call plus a manifest (seed, sha256 of the routing tensors)."""
    inp = make_routing_inputs(cfg, zipf_scale)
    inp.update(make_expert_weights(cfg, weights_device))
    manifest = {"config": cfg.as_dict(),
                "sha256": {k: _sha(v) for k, v in inp.items()
                           if v is not None and k in ("x", "W_g", "bias", "u")}}
    inp["manifest"] = manifest
    return inp


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bytes (copied to the host)."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
