"""Router kernel (moe_route) against the oracle router on the same bf16 bytes."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_moe_layer_route_gb300 as M
import workloads as W
from moe_harness import f64, GATE_ATOL

pytestmark = pytest.mark.gpu

CASES = [  # T, d, E, k, mode, bias
    (1, 64, 1, 1, W.PLAIN, "zero"),
    (37, 64, 3, 2, W.PLAIN, "zero"),
    (300, 256, 8, 2, W.PLAIN, "zero"),
    (1000, 512, 16, 2, W.GUMBEL, "zero"),
    (777, 2048, 64, 6, W.BIAS_SELECT, "normal"),
    (513, 1024, 128, 2, W.BIAS_SELECT, "zipf"),
    (200, 128, 256, 8, W.PLAIN, "zero"),
    (64, 192, 100, 5, W.GUMBEL, "zero"),
    (96, 128, 8, 8, W.BIAS_SELECT, "normal"),
    # experts per lane of the selection warp: one lane of two (33), three (96), seven (200)
    (333, 256, 33, 3, W.BIAS_SELECT, "normal"),
    (250, 256, 96, 4, W.GUMBEL, "zero"),
    (130, 192, 200, 7, W.BIAS_SELECT, "zipf"),
    # Gumbel draws of E = 33 per row: every other token's row starts off an 8-byte boundary, so
    # the selection's two-float runs of u alternate between vector and scalar loads
    (201, 128, 33, 2, W.GUMBEL, "zero"),
]


def run_route(cfg, inp, prepared=False):
    """moe_route; prepared: with the router weights transposed once by moe_prepare_router."""
    mc = M.MoeConfig.from_layer(cfg)
    dev = "cuda"
    x, W_g = inp["x"].to(dev), inp["W_g"].to(dev)
    bias = inp["bias"].to(dev)
    u = inp["u"].to(dev) if inp["u"] is not None else None
    idx = torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device=dev)
    w = torch.full((cfg.T, cfg.k), float("nan"), dtype=torch.float32, device=dev)
    ws = M.alloc_workspace(mc)
    M.route(mc, x, W_g, bias, u, idx, w, ws, W_g_t=M.prepare_router(W_g) if prepared else None)
    assert M.device_status(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy()


def oracle_for(cfg, inp):
    u = inp["u"].numpy() if inp["u"] is not None else None
    return O.route(f64(inp["x"]), f64(inp["W_g"]), cfg.k, cfg.mode,
                   inp["bias"].double().numpy(), u, cfg.tau, cfg.n_groups, cfg.topk_groups)


@pytest.mark.parametrize("T,d,E,k,mode,bias", CASES)
def test_route_matches_oracle(T, d, E, k, mode, bias):
    cfg = W.small_config(T=T, d=d, E=E, k=k, f=64, mode=mode, tau=0.5 if mode == W.GUMBEL else 1.0,
                         seed=T + E, bias=bias, bias_var=0.1)
    inp = W.make_routing_inputs(cfg, zipf_scale=0.8 if bias == "zipf" else None)
    idx, w = run_route(cfg, inp)
    r = oracle_for(cfg, inp)
    exempt = r["margin"] < O.TIE_MARGIN
    diff = (idx != r["topk_idx"]).any(1)
    assert not (diff & ~exempt).any(), np.nonzero(diff & ~exempt)[0][:10]
    w_ref = O.gates(r["logits"], r["scores"], idx, mode)
    assert np.abs(w - w_ref).max() <= GATE_ATOL
    np.testing.assert_allclose(w.sum(1), 1.0, atol=2e-6)
    # the once-prepared transpose gives the same bits as the per-call one
    idx_p, w_p = run_route(cfg, inp, prepared=True)
    assert np.array_equal(idx_p, idx) and np.array_equal(w_p.view(np.uint32), w.view(np.uint32))


def test_route_exact_ties_lowest_index():
    """Duplicated router columns give bit-identical logits on both sides; the lower index must
    win every such tie, in the same order as the oracle."""
    cfg = W.small_config(T=512, d=256, E=16, k=4, f=64, seed=21)
    inp = W.make_routing_inputs(cfg)
    Wg = inp["W_g"].clone()
    for dst, src in ((3, 1), (7, 1), (12, 5), (15, 0)):
        Wg[:, dst] = Wg[:, src]
    inp["W_g"] = Wg
    idx, w = run_route(cfg, inp)
    r = oracle_for(cfg, inp)
    s = -np.sort(-r["scores"], 1)[:, : cfg.k + 1]
    gaps = s[:, :-1] - s[:, 1:]
    near = ((gaps > 0) & (gaps < O.TIE_MARGIN)).any(1)      # inexact near-ties stay exempt
    same = (idx == r["topk_idx"]).all(1)
    assert (same | near).all()
    n_exact_tie_tokens = ((gaps == 0).any(1) & ~near).sum()
    assert n_exact_tie_tokens > 50                           # the ties were really exercised


def test_route_k_equals_E_zero_router():
    """W_g = 0: every score ties, so the order is 0..E-1 and every gate is 1/E."""
    cfg = W.small_config(T=70, d=128, E=6, k=6, f=64, seed=3)
    inp = W.make_routing_inputs(cfg)
    inp["W_g"] = torch.zeros_like(inp["W_g"])
    idx, w = run_route(cfg, inp)
    assert (idx == np.arange(6)[None, :]).all()
    np.testing.assert_allclose(w, 1.0 / 6, atol=1e-7)


def test_route_near_ties_are_decided_exactly():
    """Two router columns that differ in one weight by 16 bf16 ulps give logit differences
    ~N(0, 3e-5): many lie above the 1e-5 exemption yet inside the router's near-tie band (8e-6
    times the row's largest |logit| at d = 2048, and the pair's column is scaled to give logits
    of a few units), where the token is re-decided from plain fp32 dot products. It must pick
    and order them exactly as the oracle does."""
    cfg = W.small_config(T=2048, d=2048, E=64, k=4, f=64, seed=31)
    inp = W.make_routing_inputs(cfg)
    Wg = inp["W_g"].float()
    Wg[:, 2] *= 3.0                      # make the pair likely to be inside the top-(k+1)
    Wg[:, 5] = Wg[:, 2]
    Wg[100, 2] = 2.0 ** -12
    Wg[100, 5] = 2.0 ** -12 + 16 * 2.0 ** -19
    inp["W_g"] = Wg.to(torch.bfloat16)
    assert float(inp["W_g"][100, 5].float() - inp["W_g"][100, 2].float()) == 16 * 2.0 ** -19
    idx, w = run_route(cfg, inp)
    r = oracle_for(cfg, inp)
    exempt = r["margin"] < O.TIE_MARGIN
    both = np.isin(r["topk_idx"], [2, 5]).sum(1) == 2
    close = both & ~exempt
    assert close.sum() > 100             # many non-exempt near-ties were exercised
    diff = (idx != r["topk_idx"]).any(1)
    assert not (diff & ~exempt).any(), np.nonzero(diff & ~exempt)[0][:10]


GROUP_CASES = [  # T, d, E, k, mode, bias, n_groups, topk_groups
    (1000, 1024, 64, 6, W.BIAS_SELECT, "normal", 8, 3),
    (513, 2048, 256, 8, W.BIAS_SELECT, "normal", 8, 4),
    (300, 256, 64, 2, W.PLAIN, "zero", 8, 1),
    (700, 512, 16, 2, W.GUMBEL, "zero", 4, 2),
    (129, 128, 12, 3, W.PLAIN, "zero", 3, 3),       # every group kept: plain top-k
    (64, 192, 64, 4, W.PLAIN, "zero", 64, 4),       # one expert per group: plain top-k
]


@pytest.mark.parametrize("T,d,E,k,mode,bias,G,Gk", GROUP_CASES)
def test_group_limited_route_matches_oracle(T, d, E, k, mode, bias, G, Gk):
    cfg = W.small_config(T=T, d=d, E=E, k=k, f=64, mode=mode, tau=0.5 if mode == W.GUMBEL else 1.0,
                         seed=T + E + G, bias=bias, bias_var=0.1, n_groups=G, topk_groups=Gk)
    inp = W.make_routing_inputs(cfg)
    idx, w = run_route(cfg, inp)
    r = oracle_for(cfg, inp)
    exempt = r["margin"] < O.TIE_MARGIN
    diff = (idx != r["topk_idx"]).any(1)
    assert not (diff & ~exempt).any(), np.nonzero(diff & ~exempt)[0][:10]
    # every selected expert lies in one of the token's topk_groups kept groups
    assert (np.array([len(set(row)) for row in (idx // (E // G))]) <= Gk).all()
    w_ref = O.gates(r["logits"], r["scores"], idx, mode)
    assert np.abs(w - w_ref).max() <= GATE_ATOL


def test_group_near_ties_are_decided_exactly():
    """The best experts of groups 0 and 1 are two router columns 16 bf16 ulps apart in one
    weight, so the group decision of many tokens hangs on a logit difference inside the router's
    near-tie band yet above the exemption margin. The full exact recompute must decide it."""
    cfg = W.small_config(T=2048, d=2048, E=32, k=2, f=64, seed=41, n_groups=4, topk_groups=1)
    inp = W.make_routing_inputs(cfg)
    Wg = inp["W_g"].float()
    Wg[:, 3] *= 3.0
    Wg[:, 8 + 4] = Wg[:, 3]
    Wg[100, 3] = 2.0 ** -12
    Wg[100, 8 + 4] = 2.0 ** -12 + 16 * 2.0 ** -19
    inp["W_g"] = Wg.to(torch.bfloat16)
    idx, w = run_route(cfg, inp)
    r = oracle_for(cfg, inp)
    exempt = r["margin"] < O.TIE_MARGIN
    s = f64(inp["x"]) @ f64(inp["W_g"])
    gs = np.sort(s.reshape(cfg.T, 4, 8).max(2), 1)
    top_is_pair = (np.abs(s[:, 3] - s[:, 12]) < 1e-4) & (np.maximum(s[:, 3], s[:, 12]) == gs[:, -1])
    assert (top_is_pair & ~exempt).sum() > 100     # many non-exempt group near-ties exercised
    diff = (idx != r["topk_idx"]).any(1)
    assert not (diff & ~exempt).any(), np.nonzero(diff & ~exempt)[0][:10]


def test_route_zero_columns_tie_lowest_index():
    """All-zero router columns give logits of exactly zero on both sides (every product is a
    signed zero), so those experts tie at score 0 in PLAIN mode; the lower index must win, in the
    oracle's order, wherever they reach the top-k."""
    cfg = W.small_config(T=400, d=256, E=12, k=5, f=64, seed=5)
    inp = W.make_routing_inputs(cfg)
    Wg = inp["W_g"].clone()
    for c in (2, 5, 6, 11):
        Wg[:, c] = 0
    inp["W_g"] = Wg
    idx, w = run_route(cfg, inp)
    r = oracle_for(cfg, inp)
    s = -np.sort(-r["scores"], 1)[:, : cfg.k + 1]
    gaps = s[:, :-1] - s[:, 1:]
    inexact = ((gaps > 0) & (gaps < O.TIE_MARGIN)).any(1)   # inexact near-ties stay exempt
    same = (idx == r["topk_idx"]).all(1)
    assert (same | inexact).all(), np.nonzero(~(same | inexact))[0][:10]
    zero_picked = np.isin(r["topk_idx"], (2, 5, 6, 11)).sum(1)
    assert (zero_picked >= 2).sum() > 20       # zero-score ties were really decided


def test_route_unaligned_bias_and_noise_same_bits():
    """The selection loads a lane's run of biases (or Gumbel draws) as vectors when the run is
    whole and aligned, else element by element. Views one float off their allocation's alignment
    must give the same bits as aligned copies, and the oracle's selection."""
    for mode, E, bias_kind in ((W.BIAS_SELECT, 128, "normal"), (W.GUMBEL, 64, "zero")):
        cfg = W.small_config(T=300, d=256, E=E, k=2, f=64, mode=mode,
                             tau=0.5 if mode == W.GUMBEL else 1.0, seed=61 + E, bias=bias_kind,
                             bias_var=0.1)
        inp = W.make_routing_inputs(cfg)
        idx, w = run_route(cfg, inp)
        # device copies one float past a 256-byte-aligned allocation
        dev = {"bias": torch.cat([torch.zeros(1), inp["bias"]]).cuda()[1:]}
        if inp["u"] is not None:
            dev["u"] = torch.cat([torch.zeros(1), inp["u"].reshape(-1)]).cuda()[1:].view(cfg.T, E)
        assert dev["bias"].data_ptr() % 16 == 4
        idx_s, w_s = run_route_device(cfg, inp, dev)
        assert np.array_equal(idx_s, idx)
        assert np.array_equal(w_s.view(np.uint32), w.view(np.uint32))
        r = oracle_for(cfg, inp)
        exempt = r["margin"] < O.TIE_MARGIN
        assert not ((idx_s != r["topk_idx"]).any(1) & ~exempt).any()


def run_route_device(cfg, inp, dev_bias_u):
    """run_route with the bias and Gumbel draws given as (possibly offset) device views."""
    mc = M.MoeConfig.from_layer(cfg)
    dev = "cuda"
    x = inp["x"].to(dev)
    W_g = inp["W_g"].to(dev)
    idx = torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device=dev)
    w = torch.full((cfg.T, cfg.k), float("nan"), dtype=torch.float32, device=dev)
    ws = M.alloc_workspace(mc)
    M.route(mc, x, W_g, dev_bias_u["bias"], dev_bias_u.get("u"), idx, w, ws)
    assert M.device_status(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy()

