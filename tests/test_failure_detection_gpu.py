"""Failure detection on the device: every wait in the library's kernels is bounded, and a wait
that runs out records MOE_DEVFAULT_PIPELINE_TIMEOUT in the workspace's status word and returns,
leaving the context usable. moe_check_bounded_waits runs both kinds of wait (the tensor-core
pipelines' mbarrier wait, and the overflow re-route's grid barrier with one CTA skipping its
arrival) against conditions nothing will make true, with a 1 ms limit. Nothing faults, traps or
hangs: each wait ends by its own timer. The serving-side analogue in the source pages is the
overflow circuit breaker of "参数规模与稀疏激活的真相拆解", §3.2."""
import time

import pytest
import torch

import sparse_moe_layer_route_gb300 as M
import workloads as W
from moe_harness import run_layer, check_layer, to_device

pytestmark = pytest.mark.gpu


def test_bounded_waits_run_out_report_and_return():
    cfg = W.small_config(T=256, d=256, E=8, k=2, f=256, S=1, mode=W.BIAS_SELECT, bias="normal",
                         bias_var=0.1, capacity_factor=1.0, reroute=True, seed=91)
    ws = M.alloc_workspace(M.MoeConfig.from_layer(cfg))
    for _ in range(2):                     # twice: the check leaves its barrier counter clean
        expired = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        M.check_bounded_waits(1_000_000, expired, ws)
        status = M.device_status(ws)       # synchronises, reads and clears the status word
        dt = time.perf_counter() - t0
        assert status == M.DEVFAULT_PIPELINE_TIMEOUT
        assert expired.tolist() == [1, 1]  # both waits gave up
        assert dt < 0.5, dt                # after about the 1 ms limit, not the layer's 2 s
    assert M.device_status(ws) == 0
    # the context still runs a layer, with the re-route's grid barrier, correctly
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    rep = check_layer(cfg, inp, run_layer(cfg, inp))
    assert rep["n_kept"] > 0
