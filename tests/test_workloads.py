"""The seeded input generator: deterministic, right shapes and types, u inside (0, 1)."""
import numpy as np
import torch

import workloads as W


def test_tiny_inputs_deterministic_and_shaped():
    cfg = W.CONFIGS["tiny"]
    a = W.make_inputs(cfg)
    b = W.make_inputs(cfg)
    assert a["manifest"] == b["manifest"]
    assert a["x"].shape == (128, 256) and a["x"].dtype == torch.bfloat16
    assert a["W_g"].shape == (256, 8)
    assert a["W_gate"].shape == (8, 256, 512) and a["W_down"].shape == (8, 512, 256)
    assert torch.equal(a["W_up"], b["W_up"])
    assert a["u"] is None and float(a["bias"].abs().sum()) == 0.0


def test_gumbel_u_range_and_bias_recipes():
    cfg = W.small_config(T=256, d=64, E=16, k=2, f=64, mode=W.GUMBEL, tau=0.5, seed=4)
    u = W.make_routing_inputs(cfg)["u"]
    assert u.dtype == torch.float32 and float(u.min()) >= 2 ** -24 and float(u.max()) < 1.0
    cfg = W.small_config(E=64, bias="normal", bias_var=0.1, seed=1, mode=W.BIAS_SELECT)
    b = W.make_routing_inputs(cfg)["bias"]
    assert 0.15 < float(b.std()) < 0.5
    cfg = W.small_config(E=128, bias="zipf", mode=W.BIAS_SELECT)
    b = W.make_routing_inputs(cfg, zipf_scale=1.0)["bias"].double()
    lp = W.zipf_log_pmf(128, 1.1)
    assert torch.allclose(torch.sort(b, descending=True).values, lp.float().double(), atol=1e-6)


def test_skew_scale_recorded():
    assert 0.1 < W.skew_scale() < 8.0


def test_bf16_bits_view():
    t = torch.tensor([1.0, -2.0], dtype=torch.bfloat16)
    assert W.bf16_bits(t).tolist() == [0x3F80, 0xC000]
    assert W.bf16_bits(t).dtype == np.uint16
