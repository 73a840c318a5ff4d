"""The aux-loss-free bias update (moe_bias_update) against the oracle's update rule, on random
loads and on the loads of a real routed forward pass."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_moe_layer_route_gb300 as M
import workloads as W
from moe_harness import run_layer, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("E", [1, 8, 64, 256])
def test_bias_update_matches_oracle(E):
    rng = np.random.default_rng(E)
    counts = rng.integers(0, 500, size=E).astype(np.int32)
    bias = rng.standard_normal(E).astype(np.float32)
    c_d = torch.as_tensor(counts, device="cuda")
    b_d = torch.as_tensor(bias, device="cuda")
    M.bias_update(c_d, b_d)
    want = O.bias_update(bias.astype(np.float64), counts)
    np.testing.assert_allclose(b_d.cpu().numpy(), want, rtol=0, atol=2e-7 * (1 + np.abs(want).max()))


def test_bias_update_zero_load_and_custom_rates():
    counts = torch.zeros(16, dtype=torch.int32, device="cuda")
    b = torch.full((16,), 0.5, dtype=torch.float32, device="cuda")
    M.bias_update(counts, b, decay=0.9, rate=0.05)   # mean 0: ratio 0, only the decay applies
    assert torch.allclose(b, torch.full_like(b, 0.45))


def test_bias_update_after_routed_forward():
    cfg = W.small_config(T=1024, d=256, E=32, k=4, f=128, mode=W.BIAS_SELECT, bias="normal",
                         bias_var=0.1, capacity_factor=1.0, seed=44)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    gpu = run_layer(cfg, inp)
    counts = gpu["counts"]
    assert counts.sum() == cfg.T * cfg.k            # loads are pre-capacity selections
    b = inp["bias"].clone()
    M.bias_update(torch.as_tensor(counts, device="cuda"), b)
    want = O.bias_update(inp["bias"].double().cpu().numpy(), counts)
    np.testing.assert_allclose(b.cpu().numpy(), want, rtol=0, atol=1e-6)
