"""Level-2 overflow re-route on the GPU against the oracle's slot-order walk, through the C ABI:
the whole layer (final experts, gates, dispatch, output) and the standalone entry point."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_moe_layer_route_gb300 as M
import workloads as W
from moe_harness import run_layer, check_layer, to_device, oracle_route, f64

pytestmark = pytest.mark.gpu

CASES = [
    dict(T=1024, d=256, E=32, k=2, f=128, mode=W.BIAS_SELECT, bias="zipf", capacity_factor=1.0),
    dict(T=700, d=128, E=8, k=2, f=128, mode=W.PLAIN, capacity_factor=0.5),   # most stay dropped
    dict(T=1000, d=512, E=16, k=2, f=128, mode=W.GUMBEL, tau=0.5, capacity_factor=1.0),
    dict(T=300, d=128, E=4, k=3, f=64, S=1, mode=W.PLAIN, capacity_factor=1.0),  # few choices left
    dict(T=37, d=64, E=3, k=2, f=64, mode=W.PLAIN, capacity_factor=1.0),        # ragged, tiny
    dict(T=4096, d=1024, E=64, k=6, f=128, S=2, mode=W.BIAS_SELECT, bias="zipf",
         capacity_factor=1.25),
    dict(T=600, d=256, E=256, k=8, f=64, mode=W.BIAS_SELECT, bias="zipf", capacity_factor=1.0),
]


@pytest.mark.parametrize("kw", CASES, ids=[f"rr{i}" for i in range(len(CASES))])
def test_reroute_layer_matches_oracle(kw):
    cfg = W.small_config(seed=kw["T"] + kw["E"] + 7, reroute=True, **kw)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda",
                                  zipf_scale=1.5 if kw.get("bias") == "zipf" else None))
    gpu = run_layer(cfg, inp)
    rep = check_layer(cfg, inp, gpu)
    assert rep["reroute_first_diff"] == -1 or rep["exempt"] >= 0
    if kw["capacity_factor"] >= 1.0:
        assert rep["rerouted_slots"] > 0                # the re-route really ran


def test_reroute_fills_capacity_that_level1_leaves_empty():
    """Every token prefers two experts: Level 1 fills them and drops the rest; Level 2 must use
    the other experts' room, up to the total capacity."""
    cfg = W.small_config(T=512, d=128, E=8, k=2, f=64, seed=5, capacity_factor=1.0, reroute=True)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    Wg = inp["W_g"].float()
    Wg[:, 0] += 0.5
    Wg[:, 1] += 0.45
    inp["W_g"] = Wg.to(torch.bfloat16)
    inp["x"] = (inp["x"].float().abs() * 0.3 + 0.2).to(torch.bfloat16)
    gpu = run_layer(cfg, inp)
    rep = check_layer(cfg, inp, gpu)
    # C = 128 per expert x 8 = room for every slot; a slot whose token already uses every expert
    # that still has room stays dropped (the oracle agrees, checked above)
    assert rep["n_kept"] >= 0.95 * 512 * 2
    assert rep["rerouted_slots"] > 500


def test_reroute_exact_ties_and_near_ties_in_preferences():
    """Duplicated router columns (exact ties, the lower index first) and a pair 16 bf16 ulps apart
    (inside the tensor core's error, above the exemption) among the fallback experts."""
    cfg = W.small_config(T=2048, d=2048, E=16, k=2, f=64, seed=11, mode=W.BIAS_SELECT,
                         bias="normal", bias_var=0.1, capacity_factor=1.0, reroute=True)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    b = inp["bias"].clone()
    b[0] += 2.0                                       # experts 0, 1 hot: most of their slots drop
    b[1] += 2.0
    inp["bias"] = b
    Wg = inp["W_g"].float()
    Wg[:, 9] = Wg[:, 4]                               # exact ties
    Wg[:, 12] = Wg[:, 6]                              # near-ties: one weight 16 ulps apart
    Wg[100, 6] = 2.0 ** -12
    Wg[100, 12] = 2.0 ** -12 + 16 * 2.0 ** -19
    inp["W_g"] = Wg.to(torch.bfloat16)
    b2 = inp["bias"].clone()
    b2[12] = b2[6]
    b2[9] = b2[4]
    inp["bias"] = b2
    gpu = run_layer(cfg, inp)
    rep = check_layer(cfg, inp, gpu)
    assert rep["rerouted_slots"] > 500


def test_standalone_entry_points_compose():
    """moe_route -> moe_permute -> moe_overflow_reroute -> moe_permute gives the layer's routing."""
    cfg = W.small_config(T=1024, d=256, E=32, k=2, f=128, mode=W.BIAS_SELECT, bias="zipf",
                         capacity_factor=1.0, seed=3, reroute=True)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda", zipf_scale=1.5))
    gpu = run_layer(cfg, inp)
    mc = M.MoeConfig.from_layer(cfg)
    dev = inp["x"].device
    T, k, E = cfg.T, cfg.k, cfg.E
    i32 = dict(dtype=torch.int32, device=dev)
    idx = torch.empty((T, k), **i32)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    counts = torch.empty(E, **i32)
    offsets = torch.empty(E + 1, **i32)
    perm_slot = torch.empty(T * k, **i32)
    slot_pos = torch.empty(T * k, **i32)
    ws = M.alloc_workspace(mc, dev)
    M.route(mc, inp["x"], inp["W_g"], inp["bias"], None, idx, w, ws)
    M.permute(mc, idx, counts, offsets, perm_slot, slot_pos, ws)
    M.overflow_reroute(mc, inp["x"], inp["bias"], None, idx, w, counts, slot_pos, ws)
    M.permute(mc, idx, counts, offsets, perm_slot, slot_pos, ws)
    assert M.device_status(ws) == 0
    assert np.array_equal(idx.cpu().numpy(), gpu["topk_idx"])
    assert np.array_equal(w.cpu().numpy(), gpu["topk_w"])
    for key, t in (("counts", counts), ("offsets", offsets), ("perm_slot", perm_slot),
                   ("slot_pos", slot_pos)):
        assert np.array_equal(t.cpu().numpy(), gpu[key]), key


def test_reroute_is_deterministic():
    cfg = W.small_config(T=4096, d=512, E=64, k=6, f=64, mode=W.BIAS_SELECT, bias="zipf",
                         capacity_factor=1.0, seed=8, reroute=True)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda", zipf_scale=1.5))
    a = run_layer(cfg, inp)
    b = run_layer(cfg, inp)
    for key in ("topk_idx", "topk_w", "perm_slot", "slot_pos"):
        assert np.array_equal(a[key], b[key]), key
    assert torch.equal(a["out_t"], b["out_t"])


def test_reroute_full_size_skewed_prefill():
    """The skewed prefill workload (T=16384, d=7168, E=128, k=2, C=320) with the re-route: final
    experts against the oracle walk on every token, the output on a seeded sample of tokens
    (re-routed ones among them)."""
    import dataclasses
    cfg = dataclasses.replace(W.CONFIGS["skewed_cap"], reroute=True)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    gpu = run_layer(cfg, inp)
    x64, r = oracle_route(cfg, inp)
    rng = np.random.default_rng(cfg.seed)
    moved = np.nonzero((gpu["topk_idx"] != gpu["primary_idx"]).any(1))[0]
    toks = set(rng.choice(cfg.T, size=16, replace=False).tolist()) | {0, cfg.T - 1}
    toks |= set(moved[:: max(1, moved.size // 8)][:8].tolist())
    rep = check_layer(cfg, inp, gpu, tokens=sorted(toks), x64=x64, r=r)
    print(rep)
    assert rep["C"] == 320 and rep["rerouted_slots"] > 10000
    assert rep["n_kept"] > 30000                     # Level 1 alone keeps about 10-14 K
