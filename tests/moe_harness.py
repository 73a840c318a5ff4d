"""Shared helpers of the parity tests: run the CUDA layer through the C ABI, run the oracle on the
same bytes, and compare under the parity contract.

Contract (per token):
  * expert indices bit-exact, except tokens whose oracle top-(k+1) adjacent score gap is below
    1e-5 (exempt; counted and reported);
  * gates within 1e-5 of the oracle's gates at the GPU's indices (the contract's gate
    tolerance; the router's logits are within about 2e-6 of the exact ones, and a softmax
    over the selected logits moves by at most half the error of a logit difference, doubled by
    1/tau = 2 for Gumbel scores);
  * counts / offsets / perm_slot / slot_pos bit-exact against the oracle dispatch run on the
    GPU's indices;
  * layer output (bf16) against the oracle's float64 output conditioned on the GPU's indices:
    max-abs <= 2e-2 and relative L2 <= 1e-2 (with quantized experts, the oracle runs on its own
    quantize-dequantize of the same bf16 weights).
  * with the Level-2 overflow re-route: the router's own indices (before the re-route) follow
    the rule above; the oracle's re-route walk, run on those indices, must give the GPU's final
    indices, unless the first token where they differ had an oracle re-route decision gap below
    1e-5 (a near-tie, counted; everything after it is compared conditioned on the GPU's final
    indices, as above).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import sparse_moe_layer_route_gb300 as M
import workloads as W

GATE_ATOL = 1e-5
OUT_MAXABS = 2e-2
OUT_RELL2 = 1e-2


def bits(t):
    return W.bf16_bits(t)


def f64(t):
    return O.bf16_bits_to_f64(bits(t))


def to_device(inp, dev="cuda"):
    out = {}
    for k, v in inp.items():
        out[k] = v.to(dev) if isinstance(v, torch.Tensor) else v
    return out


def pack_down(inp):
    """fp16 re-encodings of the down weights for the fp16 down path (one-time preparation)."""
    if "W_down_f16" not in inp:
        inp["W_down_f16"] = M.packed_f16(inp["W_down"])
        inp["Ws_down_f16"] = M.packed_f16(inp["Ws_down"]) if inp.get("Ws_down") is not None \
            else None
    return inp


def quantize_inputs(inp, bits):
    """GPU group-wise quantization of every expert matrix (one-time weight preparation)."""
    key = f"q{bits}"
    if key not in inp:
        names = ("W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down")
        qs = {n: (M.quantize_weights(inp[n], bits) if inp.get(n) is not None else None)
              for n in names}
        inp[key] = qs
        inp[key + "_struct"] = M.make_qweights(*[qs[n] for n in names])
    return inp[key], inp[key + "_struct"]


def prepare_router(inp):
    """The router weights transposed once (moe_prepare_router), as a deployment would."""
    if "W_g_t" not in inp:
        inp["W_g_t"] = M.prepare_router(inp["W_g"])
    return inp["W_g_t"]


def run_layer(cfg, inp, capacity_override=0, stream=None, f16=True, prepared=True):
    """moe_layer_forward with every routing output requested; returns numpy arrays.
    f16: use the fp16 down path (W_down re-encoded once), else the bf16 down path.
    prepared: pass the router weights transposed once (else each call transposes them).
    With cfg.weight_bits the experts are quantized on the GPU first."""
    mc = M.MoeConfig.from_layer(cfg)
    mc.capacity_override = capacity_override
    T, k, E, d = cfg.T, cfg.k, cfg.E, cfg.d
    dev = inp["x"].device
    i32 = dict(dtype=torch.int32, device=dev)
    idx = torch.full((T, k), -7, **i32)
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
    counts = torch.full((E,), -7, **i32)
    offsets = torch.full((E + 1,), -7, **i32)
    perm_slot = torch.full((T * k,), -7, **i32)
    slot_pos = torch.full((T * k,), -7, **i32)
    out = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = M.alloc_workspace(mc, dev)
    bits = getattr(cfg, "weight_bits", 0)
    wgt = prepare_router(inp) if prepared else None
    if bits:
        _, qstruct = quantize_inputs(inp, bits)
        weights = M.make_weights(inp["W_g"], inp["bias"], None, None, None, quant=qstruct,
                                 W_g_t=wgt)
    else:
        if f16:
            pack_down(inp)
        weights = M.make_weights(inp["W_g"], inp["bias"], inp["W_gate"], inp["W_up"],
                                 inp["W_down"], inp.get("Ws_gate"), inp.get("Ws_up"),
                                 inp.get("Ws_down"), inp.get("W_down_f16") if f16 else None,
                                 inp.get("Ws_down_f16") if f16 else None, W_g_t=wgt)
    ro = M.make_route_out(idx, w, counts, offsets, perm_slot, slot_pos)
    primary = None
    if getattr(cfg, "reroute", False):
        # the router's own choice, before the re-route (deterministic: the layer computes the same)
        p_idx = torch.empty((T, k), **i32)
        p_w = torch.empty((T, k), dtype=torch.float32, device=dev)
        M.route(mc, inp["x"], inp["W_g"], inp["bias"], inp.get("u"), p_idx, p_w, ws, stream,
                W_g_t=wgt)
        primary = p_idx.cpu().numpy()
    M.layer_forward(mc, weights, inp["x"], inp.get("u"), out, ro, ws, stream)
    status = M.device_status(ws, stream)
    res = {"topk_idx": idx.cpu().numpy(), "topk_w": w.cpu().numpy(),
           "counts": counts.cpu().numpy(), "offsets": offsets.cpu().numpy(),
           "perm_slot": perm_slot.cpu().numpy(), "slot_pos": slot_pos.cpu().numpy(),
           "out_t": out, "status": status, "ws": ws, "primary_idx": primary}
    return res


def _oracle_weights(mats, bits):
    """bf16 matrices widened, or (bits > 0) the oracle's own quantize-dequantize of them."""
    ws = tuple(f64(m) for m in mats)
    if bits:
        ws = tuple(O.dequantize_groupwise(*O.quantize_groupwise(w, bits)) for w in ws)
    return ws


def expert_getter(inp, bits=0):
    def get(e):
        return _oracle_weights((inp["W_gate"][e], inp["W_up"][e], inp["W_down"][e]), bits)
    return get


def shared_getter(inp, bits=0):
    def get(s):
        return _oracle_weights((inp["Ws_gate"][s], inp["Ws_up"][s], inp["Ws_down"][s]), bits)
    return get


def oracle_route(cfg, inp):
    x64 = f64(inp["x"])
    Wg64 = f64(inp["W_g"])
    bias = inp["bias"].double().cpu().numpy() if inp["bias"] is not None else None
    u = inp["u"].cpu().numpy() if inp.get("u") is not None else None
    r = O.route(x64, Wg64, cfg.k, cfg.mode, bias, u, cfg.tau, cfg.n_groups, cfg.topk_groups)
    return x64, r


def check_layer(cfg, inp, gpu, tokens=None, capacity_override=0, x64=None, r=None,
                out_scale=1.0):
    """Assert the parity contract; returns a report dict. out_scale: a power of two both outputs
    are divided by (exactly) before the output bounds apply, for layers whose outputs are far
    from unit scale."""
    if r is None:
        x64, r = oracle_route(cfg, inp)
    T, k, E = cfg.T, cfg.k, cfg.E
    assert gpu["status"] == 0, f"device status {gpu['status']:#x}"
    exempt = r["margin"] < O.TIE_MARGIN
    idx_g = gpu["topk_idx"]
    assert idx_g.min() >= 0 and idx_g.max() < E
    C = O.capacity(T, k, E, cfg.capacity_factor, capacity_override)
    idx_p = gpu["primary_idx"] if gpu.get("primary_idx") is not None else idx_g
    flipped = (idx_p != r["topk_idx"]).any(axis=1)
    bad = np.nonzero(flipped & ~exempt)[0]
    assert bad.size == 0, f"{bad.size} non-exempt tokens routed differently, e.g. {bad[:5]}"
    rr_report = {}
    if gpu.get("primary_idx") is not None and C is not None:
        rr = O.overflow_reroute(idx_p, O.permute(idx_p, E, C)["slot_pos"], r["scores"], E, C)
        diff = (idx_g != rr["topk_idx"]).any(axis=1)
        first = int(np.argmax(diff)) if diff.any() else -1
        if first >= 0:
            assert rr["margin"][first] < O.TIE_MARGIN, \
                f"re-route differs first at token {first} (decision gap {rr['margin'][first]})"
        rr_report = {"rerouted_slots": int(rr["rerouted"].sum()), "reroute_first_diff": first}
    w_cond = O.gates(r["logits"], r["scores"], idx_g, cfg.mode)
    gerr = np.abs(gpu["topk_w"] - w_cond).max()
    assert gerr <= GATE_ATOL, f"gate error {gerr}"
    p = O.permute(idx_g, E, C)
    for key in ("counts", "offsets", "perm_slot", "slot_pos"):
        assert np.array_equal(gpu[key], p[key]), f"{key} differs from the oracle dispatch"
    bits = getattr(cfg, "weight_bits", 0)
    out_ref, _ = O.layer_from_routing(x64, idx_g, w_cond, E, C, expert_getter(inp, bits), cfg.S,
                                      shared_getter(inp, bits), tokens)
    out_t = gpu["out_t"] if tokens is None else gpu["out_t"][torch.as_tensor(tokens)]
    out_g = f64(out_t) / out_scale
    out_ref = out_ref / out_scale
    err = np.abs(out_g - out_ref)
    maxabs = float(err.max())
    rel_l2 = float(np.linalg.norm(out_g - out_ref) / max(np.linalg.norm(out_ref), 1e-30))
    assert np.isfinite(out_g).all()
    assert maxabs <= OUT_MAXABS and rel_l2 <= OUT_RELL2, (maxabs, rel_l2)
    return {"exempt": int(exempt.sum()), "flipped": int(flipped.sum()), "gate_err": float(gerr),
            "maxabs": maxabs, "rel_l2": rel_l2, "n_kept": int(p["n_kept"]), "C": C, **rr_report}
