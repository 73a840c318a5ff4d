"""fp16's range on the expert path. The fp16 down path stores the SwiGLU activations H and the
gate-scaled slot rows in fp16 (11 significant bits, but a largest finite value of 65504); the
quantized experts do too. A value past that is clamped, and the library must say so
(MOE_DEVFAULT_FP16_RANGE), never return a clamped layer output silently. The bf16 down path keeps
H in bf16 and the slot rows in fp32 (fp32's range): on the same data it must match the oracle.

Expert weights are scaled by powers of two (exact in bf16), so the router and its gates are
those of an ordinary layer while H, or only the expert outputs, leave fp16's range. SwiGLU
experts: "GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token", §3.3."""
import pytest
import torch

import sparse_moe_layer_route_gb300 as M
import workloads as W
from moe_harness import run_layer, check_layer, to_device

pytestmark = pytest.mark.gpu


def scaled_inputs(cfg, gate_up=1.0, down=1.0):
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    for key, f in (("W_gate", gate_up), ("W_up", gate_up), ("Ws_gate", gate_up),
                   ("Ws_up", gate_up), ("W_down", down), ("Ws_down", down)):
        if inp.get(key) is not None and f != 1.0:
            inp[key] = (inp[key].float() * f).to(torch.bfloat16)   # a power of two: exact
    return inp


CFG = dict(T=300, d=256, E=8, k=2, f=512, S=1, mode=W.BIAS_SELECT, bias="normal", bias_var=0.1)


@pytest.mark.parametrize("gate_up,down,out_scale", [
    (2.0 ** 8, 1.0, 2.0 ** 16),    # H = silu(G) U reaches ~2^16 and beyond: H leaves fp16's range
    (1.0, 2.0 ** 16, 2.0 ** 16),   # H ordinary, the expert outputs ~2^16 times larger
])
def test_large_activations_flagged_on_fp16_path_exact_on_bf16_path(gate_up, down, out_scale):
    cfg = W.small_config(seed=77, **CFG)
    inp = scaled_inputs(cfg, gate_up, down)
    # the fp16 re-encoding of W_down itself stays in range (|w| well below 65504)
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    inp["W_down_f16"] = M.packed_f16(inp["W_down"], fault_bits=fault)
    inp["Ws_down_f16"] = M.packed_f16(inp["Ws_down"], fault_bits=fault)
    torch.cuda.synchronize()
    assert int(fault.item()) == 0
    f16 = run_layer(cfg, inp, f16=True)
    assert f16["status"] & M.DEVFAULT_FP16_RANGE, f"status {f16['status']:#x}: clamp not reported"
    assert f16["status"] == M.DEVFAULT_FP16_RANGE          # and nothing else went wrong
    # the bf16 down path on the same bytes: no report, and the oracle's output
    bf = run_layer(cfg, inp, f16=False)
    assert bf["status"] == 0
    rep = check_layer(cfg, inp, bf, out_scale=out_scale)
    assert rep["flipped"] == 0
    # the outputs really are beyond fp16's range (the test exercises what it claims)
    assert bf["out_t"].float().abs().max().item() > 65504.0


def test_ordinary_layer_reports_nothing_on_fp16_path():
    cfg = W.small_config(seed=78, **CFG)
    inp = scaled_inputs(cfg)
    out = run_layer(cfg, inp, f16=True)
    assert out["status"] == 0
    check_layer(cfg, inp, out)


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_experts_report_fp16_clamp(bits):
    """Quantized experts carry H and the slot rows in fp16 as well."""
    cfg = W.small_config(T=64, d=256, E=16, k=2, f=256, S=1, seed=79, weight_bits=bits)
    inp = scaled_inputs(cfg, gate_up=2.0 ** 8)
    out = run_layer(cfg, inp)
    assert out["status"] == M.DEVFAULT_FP16_RANGE
    plain = run_layer(cfg, scaled_inputs(cfg))
    assert plain["status"] == 0
