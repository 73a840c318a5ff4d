"""Whole layer (moe_layer_forward) against the oracle at sizes the oracle finishes in seconds,
plus the identities that tie the entry points together."""
import numpy as np
import pytest
import torch

import sparse_moe_layer_route_gb300 as M
import workloads as W
from moe_harness import run_layer, check_layer, to_device

pytestmark = pytest.mark.gpu

SMALL = [
    dict(T=300, d=256, E=8, k=2, f=512, mode=W.PLAIN),
    dict(T=257, d=192, E=5, k=3, f=320, S=1, mode=W.BIAS_SELECT, bias="normal", bias_var=0.1),
    dict(T=1000, d=512, E=16, k=2, f=384, mode=W.GUMBEL, tau=0.5, capacity_factor=1.25),
    dict(T=2048, d=256, E=64, k=6, f=128, S=2, mode=W.BIAS_SELECT, bias="normal", bias_var=0.1),
    dict(T=1024, d=256, E=32, k=2, f=256, mode=W.BIAS_SELECT, bias="zipf", capacity_factor=1.25),
    dict(T=1, d=64, E=1, k=1, f=64),
    dict(T=100, d=128, E=4, k=4, f=128, S=1, capacity_factor=0.05),
    dict(T=200, d=128, E=256, k=8, f=64),
    dict(T=1024, d=256, E=64, k=6, f=128, S=2, mode=W.BIAS_SELECT, bias="normal", bias_var=0.1,
         n_groups=8, topk_groups=3, capacity_factor=1.0),
    # long expert segments (T*k >= 320 E): 256-row tiles on CTA pairs, odd tile counts included
    dict(T=1024, d=256, E=4, k=2, f=256, S=1),
    dict(T=700, d=512, E=4, k=2, f=384, mode=W.BIAS_SELECT, bias="normal", bias_var=0.1),
    dict(T=1500, d=256, E=8, k=3, f=128, S=2, mode=W.GUMBEL, tau=0.5),
    # rows of 2-4 column groups per combine thread (a CTA per token): with a capacity limit and
    # a shared expert (d = 2560), and without either (d = 8192)
    dict(T=400, d=2560, E=8, k=2, f=128, S=1, mode=W.BIAS_SELECT, bias="zipf",
         capacity_factor=1.0),
    dict(T=320, d=8192, E=4, k=1, f=128),
]


@pytest.mark.parametrize("kw", SMALL, ids=[f"cfg{i}" for i in range(len(SMALL))])
def test_layer_matches_oracle(kw):
    cfg = W.small_config(seed=len(kw) * 13 + kw["T"], **kw)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda",
                                  zipf_scale=1.5 if kw.get("bias") == "zipf" else None))
    gpu = run_layer(cfg, inp)
    check_layer(cfg, inp, gpu)


def test_layer_bf16_down_path():
    cfg = W.small_config(T=600, d=256, E=16, k=2, f=256, mode=W.GUMBEL, tau=0.5, seed=77)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    check_layer(cfg, inp, run_layer(cfg, inp, f16=False))


def test_layer_bf16_down_path_token_combine():
    """fp32 slot rows read by the per-token combine (d = 4096, capacity drops)."""
    cfg = W.small_config(T=512, d=4096, E=8, k=2, f=128, mode=W.BIAS_SELECT, bias="zipf",
                         capacity_factor=1.0, seed=78)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda", zipf_scale=1.5))
    check_layer(cfg, inp, run_layer(cfg, inp, f16=False))


def test_tiny_config_full():
    cfg = W.CONFIGS["tiny"]
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    rep = check_layer(cfg, inp, run_layer(cfg, inp))
    assert rep["n_kept"] == cfg.T * cfg.k


def test_layer_deterministic_and_entry_points_compose():
    cfg = W.small_config(T=700, d=256, E=16, k=3, f=256, S=1, mode=W.BIAS_SELECT,
                         bias="normal", bias_var=0.1, capacity_factor=1.1, seed=5)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    a = run_layer(cfg, inp)
    b = run_layer(cfg, inp)
    assert torch.equal(a["out_t"].view(torch.int16), b["out_t"].view(torch.int16))
    # route -> permute -> grouped_ffn -> combine gives the same bits as the fused sequence
    mc = M.MoeConfig.from_layer(cfg)
    ws = M.alloc_workspace(mc)
    dev = "cuda"
    T, k, E, d = cfg.T, cfg.k, cfg.E, cfg.d
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    M.route(mc, inp["x"], inp["W_g"], inp["bias"], None, idx, w, ws)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm_slot = torch.empty(T * k, dtype=torch.int32, device=dev)
    slot_pos = torch.empty(T * k, dtype=torch.int32, device=dev)
    M.permute(mc, idx, counts, offsets, perm_slot, slot_pos, ws)
    y = torch.empty((T * k + cfg.S * T, d), dtype=torch.float16, device=dev)
    M.grouped_ffn(mc, inp["x"], perm_slot, offsets, w, inp["W_gate"], inp["W_up"],
                  inp["W_down"], inp["Ws_gate"], inp["Ws_up"], inp["Ws_down"], y, ws,
                  W_down_f16=inp["W_down_f16"], Wsh_down_f16=inp["Ws_down_f16"])
    out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    M.combine(mc, y, slot_pos, out, ws)
    assert M.device_status(ws) == 0
    assert torch.equal(out.view(torch.int16), a["out_t"].view(torch.int16))
    assert np.array_equal(idx.cpu().numpy(), a["topk_idx"])


def test_host_buffer_entry_point_matches_device_one():
    cfg = W.small_config(T=513, d=256, E=16, k=2, f=256, mode=W.GUMBEL, tau=0.5, seed=8)
    inp_cpu = W.make_inputs(cfg, weights_device="cuda")
    inp = to_device(inp_cpu)
    ref = run_layer(cfg, inp)["out_t"]
    mc = M.MoeConfig.from_layer(cfg)
    ws = M.alloc_workspace(mc)
    weights = M.make_weights(inp["W_g"], inp["bias"], inp["W_gate"], inp["W_up"], inp["W_down"],
                             W_down_f16=inp["W_down_f16"])
    x_h = inp_cpu["x"].pin_memory()
    u_h = inp_cpu["u"].pin_memory()
    out_h = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory()
    M.layer_forward_host(mc, weights, x_h, u_h, out_h, ws)
    assert M.device_status(ws) == 0
    assert torch.equal(out_h.view(torch.int16), ref.cpu().view(torch.int16))


def _prepared(cfg, inp):
    """Config struct, weights struct, workspace and output buffer for moe_layer_forward."""
    from moe_harness import pack_down, quantize_inputs
    mc = M.MoeConfig.from_layer(cfg)
    dev = inp["x"].device
    if cfg.weight_bits:
        _, qstruct = quantize_inputs(inp, cfg.weight_bits)
        weights = M.make_weights(inp["W_g"], inp["bias"], None, None, None, quant=qstruct)
    else:
        pack_down(inp)
        weights = M.make_weights(inp["W_g"], inp["bias"], inp["W_gate"], inp["W_up"],
                                 inp["W_down"], inp.get("Ws_gate"), inp.get("Ws_up"),
                                 inp.get("Ws_down"), inp.get("W_down_f16"),
                                 inp.get("Ws_down_f16"))
    ws = M.alloc_workspace(mc, dev)
    out = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.bfloat16, device=dev)
    return mc, weights, ws, out


def test_concurrent_streams_match_serial():
    """Every piece of per-call state lives in the caller's workspace, so calls on separate
    streams and workspaces may overlap on the GPU (a serving loop does this). Layers of different
    kinds (CTA-pair GEMMs, single-CTA GEMMs with a capacity limit, the overflow re-route with its
    cooperative kernel, 8- and 4-bit experts) launched back to back on their own streams give the same
    bytes as the same calls made one at a time."""
    kinds = [
        dict(T=1024, d=256, E=4, k=2, f=256, S=1),
        dict(T=700, d=256, E=16, k=3, f=256, S=1, mode=W.BIAS_SELECT, bias="normal",
             bias_var=0.1, capacity_factor=1.1),
        dict(T=1024, d=256, E=32, k=2, f=128, mode=W.BIAS_SELECT, bias="zipf",
             capacity_factor=1.25, reroute=True),
        dict(T=96, d=256, E=8, k=2, f=256, S=1, weight_bits=8),
        # 4-bit experts: every gate/up unit is split along K, and its pieces may finish in any
        # order; their partials are still added in piece order
        dict(T=96, d=512, E=8, k=2, f=256, S=1, weight_bits=4),
    ]
    runs = []
    for i, kw in enumerate(kinds):
        cfg = W.small_config(name=f"kind{i}", seed=900 + i, **kw)
        inp = to_device(W.make_inputs(cfg, weights_device="cuda",
                                      zipf_scale=1.5 if kw.get("bias") == "zipf" else None))
        runs.append((cfg, inp) + _prepared(cfg, inp))
    serial = []
    for cfg, inp, mc, weights, ws, out in runs:
        M.layer_forward(mc, weights, inp["x"], inp.get("u"), out, None, ws)
        assert M.device_status(ws) == 0
        serial.append(out.clone())
    streams = [torch.cuda.Stream() for _ in runs]
    torch.cuda.synchronize()
    for rep in range(3):
        for (cfg, inp, mc, weights, ws, out), st in zip(runs, streams):
            out.fill_(float("nan"))
        torch.cuda.synchronize()
        for (cfg, inp, mc, weights, ws, out), st in zip(runs, streams):
            M.layer_forward(mc, weights, inp["x"], inp.get("u"), out, None, ws, st)
        torch.cuda.synchronize()
        for (cfg, inp, mc, weights, ws, out), ref in zip(runs, serial):
            assert M.device_status(ws) == 0
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), cfg.name


def test_empty_batch_clears_only_the_per_expert_outputs():
    """T = 0 launches no kernel: the dispatch outputs counts [E] and offsets [E + 1] are cleared
    (every expert receives nothing), the fault word of the allocation-free dispatch is cleared,
    the profiled layer still records all seven events, and the workspace stays clean."""
    dev, E, k = "cuda", 8, 2
    cfg = M.MoeConfig.make(0, 128, E, k, 128, n_shared=1, capacity_factor=1.0)
    ws = M.alloc_workspace(cfg)
    assert ws.numel() == 512
    i32 = dict(dtype=torch.int32, device=dev)
    empty = torch.empty((0, k), **i32)

    def filled():
        return torch.full((E,), -7, **i32), torch.full((E + 1,), -7, **i32)

    counts, offsets = filled()
    M.permute(cfg, empty, counts, offsets, empty.view(-1), empty.view(-1), ws)
    counts2, offsets2 = filled()
    fault = torch.full((1,), 99, **i32)
    M.permute_noalloc(cfg, empty, counts2, offsets2, empty.view(-1), empty.view(-1), fault)
    counts3, offsets3 = filled()
    x = torch.empty((0, 128), dtype=torch.bfloat16, device=dev)
    out = torch.empty((0, 128), dtype=torch.bfloat16, device=dev)
    Wg = torch.zeros((128, E), dtype=torch.bfloat16, device=dev)
    w = M.make_weights(Wg, None, None, None, None)      # no expert weight is read
    M.layer_forward(cfg, w, x, None, out, M.make_route_out(counts=counts3, offsets=offsets3), ws)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    M.layer_forward_profiled(cfg, w, x, None, out, None, ws, events)
    torch.cuda.synchronize()
    for c, o in ((counts, offsets), (counts2, offsets2), (counts3, offsets3)):
        assert torch.equal(c, torch.zeros_like(c)) and torch.equal(o, torch.zeros_like(o))
    assert int(fault.item()) == 0
    assert all(events[i].elapsed_time(events[i + 1]) >= 0.0 for i in range(6))
    assert M.device_status(ws) == 0
