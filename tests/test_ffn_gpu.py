"""Grouped GEMM (moe_grouped_ffn: gather, tcgen05 gate/up with SiLU*up, tcgen05 down with gate
scale + unpermute) fed the oracle's dispatch, against the oracle's per-slot SwiGLU outputs."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_moe_layer_route_gb300 as M
import workloads as W
from moe_harness import f64, expert_getter, shared_getter, OUT_MAXABS, OUT_RELL2

pytestmark = pytest.mark.gpu


def run_case(T, d, E, k, f, S, C, skew, seed, f16=True):
    cfg = W.small_config(T=T, d=d, E=E, k=k, f=f, S=S, seed=seed)
    inp = W.make_inputs(cfg, weights_device="cuda")
    rng = np.random.default_rng(seed)
    keys = rng.random((T, E))
    if skew is not None:
        keys = keys * (np.arange(1, E + 1) ** -skew)[None, :]
    idx = np.argsort(-keys, axis=1)[:, :k]
    gates = rng.random((T, k)).astype(np.float32) + 0.25
    p = O.permute(idx, E, C if C else None)
    dev = "cuda"
    mc = M.MoeConfig.make(T, d, E, k, f, n_shared=S, capacity_override=C)
    x = inp["x"].to(dev)
    # slot rows: fp16 on the fp16 down path, fp32 on the bf16 one
    y = torch.full((T * k + S * T, d), float("nan"), dtype=torch.float16 if f16 else torch.float32,
                   device=dev)
    ws = M.alloc_workspace(mc)
    Wd16 = M.packed_f16(inp["W_down"]) if f16 else None
    Wsd16 = M.packed_f16(inp["Ws_down"]) if (f16 and S > 0) else None
    M.grouped_ffn(mc, x, torch.as_tensor(p["perm_slot"], device=dev),
                  torch.as_tensor(p["offsets"], device=dev), torch.as_tensor(gates, device=dev),
                  inp["W_gate"], inp["W_up"], inp["W_down"], inp["Ws_gate"], inp["Ws_up"],
                  inp["Ws_down"], y, ws, W_down_f16=Wd16, Wsh_down_f16=Wsd16)
    assert M.device_status(ws) == 0
    x64 = f64(inp["x"])
    slot_y, shared_y = O.expert_outputs(x64, idx, p["slot_pos"], expert_getter(inp), k, None, S,
                                        shared_getter(inp))
    kept = sorted(slot_y)
    ref = np.stack([gates.reshape(-1)[s] * slot_y[s] for s in kept])
    yg = y.cpu().double().numpy()
    got = yg[kept]
    for s_i in range(S):
        ref = np.concatenate([ref, np.stack([shared_y[s_i][t] for t in range(T)])])
        got = np.concatenate([got, yg[T * k + s_i * T: T * k + (s_i + 1) * T]])
    assert np.isfinite(got).all(), "a kept row was never written"
    maxabs = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert maxabs <= OUT_MAXABS and rel <= OUT_RELL2, (maxabs, rel)
    return p


@pytest.mark.parametrize("T,d,E,k,f,S,C,skew", [
    (300, 256, 8, 2, 512, 0, 0, None),      # 128-col gate/up tiles, 256-col down tiles
    (257, 192, 5, 3, 320, 1, 0, None),      # 64-col gate/up tiles, 64-col down tiles, shared
    (2048, 128, 64, 6, 128, 2, 0, 1.0),     # 128-col down tiles, two shared experts
    (1000, 512, 16, 2, 384, 0, 150, 1.5),   # capacity drops
    (3, 64, 4, 1, 64, 0, 0, None),          # smallest shapes, 1-row segments
    (700, 256, 2, 1, 256, 0, 0, 3.0),       # one long segment (many row tiles) + a short one
    (64, 1024, 128, 2, 256, 1, 0, None),    # decode-like: most experts 0-2 rows
])
def test_grouped_ffn_matches_oracle(T, d, E, k, f, S, C, skew):
    run_case(T, d, E, k, f, S, C, skew, seed=T + d + E)


@pytest.mark.parametrize("T,d,E,k,f,S", [(300, 256, 8, 2, 512, 0), (257, 192, 5, 2, 320, 1),
                                         (129, 128, 4, 1, 128, 0)])
def test_grouped_ffn_bf16_down_path(T, d, E, k, f, S):
    """The path without the fp16 copy of W_down: H carried in bf16, down GEMM in bf16, slot rows
    in fp32."""
    run_case(T, d, E, k, f, S, 0, None, seed=T + 1, f16=False)


def test_pack_f16_matches_torch_conversion():
    g = torch.Generator(device="cuda").manual_seed(0)
    src = (torch.randn(1000003, generator=g, device="cuda") * 3).to(torch.bfloat16)
    src[:6] = torch.tensor([0.0, -0.0, 1e-6, -2.0 ** -20, 65504.0, 1.5e5], dtype=torch.bfloat16)
    dst = torch.empty(src.shape, dtype=torch.float16, device="cuda")
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.pack_f16(src, dst, fault_bits=fault)
    torch.cuda.synchronize()
    want = src.float().clamp(-65504, 65504).to(torch.float16)
    assert torch.equal(dst.view(torch.int16), want.view(torch.int16))
    assert dst[5].item() == 65504.0
    assert int(fault.item()) == M.DEVFAULT_FP16_RANGE      # 1.5e5 was clamped, and reported
    # the largest bf16 below fp16's limit converts without a report; the next one is clamped
    fault.zero_()
    ok = torch.tensor([65280.0, -65280.0, 1.0, 0.0, 2.0, 3.0, 4.0, 5.0], dtype=torch.bfloat16,
                      device="cuda")
    M.pack_f16(ok, torch.empty(8, dtype=torch.float16, device="cuda"), fault_bits=fault)
    torch.cuda.synchronize()
    assert int(fault.item()) == 0
    M.pack_f16(ok * 0 - 65536.0, torch.empty(8, dtype=torch.float16, device="cuda"),
               fault_bits=fault)
    torch.cuda.synchronize()
    assert int(fault.item()) == M.DEVFAULT_FP16_RANGE


def test_grouped_ffn_empty_experts():
    p = run_case(400, 128, 32, 1, 128, 0, 0, 4.0, seed=9)
    assert (np.diff(p["offsets"]) == 0).any()
