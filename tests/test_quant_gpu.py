"""Weight-only group-wise quantized experts on the GPU, through the C ABI: the quantizer's
scales, zero-points and codes bit-exact against the oracle's quantizer (codes read back from the
fragment layout include/moe.h documents), and the layer on quantized experts against the oracle
run on its own quantize-dequantize of the same bf16 weights."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_moe_layer_route_gb300 as M
import workloads as W
from moe_harness import run_layer, check_layer, to_device, oracle_route, f64

pytestmark = pytest.mark.gpu


def unpack_codes(q, bits, n_mat, K, N):
    """Plain [n_mat, K, N] codes from the fragment-ordered bytes (the layout of moe_qmatrix)."""
    q = q.cpu().numpy()
    m, k, n = np.meshgrid(np.arange(n_mat), np.arange(K), np.arange(N), indexing="ij")
    nt, r = n // 16, n % 16
    st, kk = k // 16, k % 16
    lane = (r % 8) * 4 + (kk % 8) // 2
    j = (kk % 2) + 2 * (r // 8) + 4 * (kk // 8)
    tile = m * (N // 16) + nt
    if bits == 8:
        off = (tile * (K // 32) + st // 2) * 512 + lane * 16 + (st % 2) * 8 + j
        return q[off]
    off = (tile * (K // 64) + st // 4) * 512 + lane * 16 + (st % 4) * 4
    words = q.view(np.uint32)[off // 4]
    return ((words >> (16 * (j % 2) + 4 * (j // 2))) & 0xF).astype(np.uint8)


def _weights_cases():
    g = torch.Generator().manual_seed(7)
    a = torch.randn(3, 256, 96, generator=g) * 0.02
    b = torch.randn(2, 384, 64, generator=g) * torch.tensor([1e-3, 50.0]).view(2, 1, 1)
    c = torch.zeros(1, 128, 32)
    c[0, :, 1] = 0.5                       # constant group
    c[0, :, 2] = -0.25
    c[0, 5, 3] = 3.0                       # a spike
    c[0, :, 4] = torch.linspace(-1, 1, 128)
    return [a, b, c]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("case", [0, 1, 2])
def test_quantizer_bit_exact(bits, case):
    Wt = _weights_cases()[case].to(torch.bfloat16)
    n_mat, K, N = Wt.shape
    qd = M.quantize_weights(Wt.cuda(), bits)
    torch.cuda.synchronize()
    q_ref, s_ref, z_ref = O.quantize_groupwise(f64(Wt), bits)
    assert np.array_equal(qd["scale"].cpu().numpy().view(np.uint16), s_ref.view(np.uint16))
    assert np.array_equal(qd["zero"].cpu().numpy(), z_ref)
    assert np.array_equal(unpack_codes(qd["q"], bits, n_mat, K, N), q_ref)


SMALL = [
    dict(T=64, d=256, E=8, k=2, f=256, S=1),
    dict(T=300, d=384, E=16, k=2, f=128, mode=W.BIAS_SELECT, bias="normal", bias_var=0.1),
    dict(T=37, d=128, E=4, k=3, f=384, S=2, capacity_factor=1.0),
    dict(T=8, d=512, E=64, k=6, f=256, S=1, mode=W.GUMBEL, tau=0.5),
    dict(T=130, d=256, E=8, k=2, f=128, capacity_factor=1.0, reroute=True),
]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("kw", SMALL, ids=[f"q{i}" for i in range(len(SMALL))])
def test_quantized_layer_matches_oracle(bits, kw):
    cfg = W.small_config(seed=kw["T"] + kw["E"] + bits, weight_bits=bits, **kw)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    gpu = run_layer(cfg, inp)
    check_layer(cfg, inp, gpu)


def test_quantized_matches_bf16_layer_closely():
    """8-bit experts move the layer output only slightly against the bf16 experts."""
    base = dict(T=64, d=512, E=8, k=2, f=256, S=1, seed=5)
    c8 = W.small_config(weight_bits=8, **base)
    c0 = W.small_config(**base)
    inp = to_device(W.make_inputs(c0, weights_device="cuda"))
    o0 = run_layer(c0, inp)["out_t"].float()
    o8 = run_layer(c8, inp)["out_t"].float()
    rel = float((o8 - o0).norm() / o0.norm())
    assert 1e-4 < rel < 3e-2, rel


def test_grouped_ffn_quantized_entry_point_matches_layer():
    cfg = W.small_config(T=96, d=256, E=8, k=2, f=256, S=1, seed=9, weight_bits=4)
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    gpu = run_layer(cfg, inp)
    mc = M.MoeConfig.from_layer(cfg)
    ws = M.alloc_workspace(mc)
    T, k, d = cfg.T, cfg.k, cfg.d
    dev = "cuda"
    perm = torch.as_tensor(gpu["perm_slot"], device=dev)
    offs = torch.as_tensor(gpu["offsets"], device=dev)
    w = torch.as_tensor(gpu["topk_w"], device=dev)
    y = torch.zeros((T * k + cfg.S * T, d), dtype=torch.float16, device=dev)
    M.grouped_ffn_quantized(mc, inp["x"], perm, offs, w, inp["q4_struct"], y, ws)
    out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    M.combine(mc, y, torch.as_tensor(gpu["slot_pos"], device=dev), out, ws)
    assert M.device_status(ws) == 0
    assert torch.equal(out, gpu["out_t"])


@pytest.mark.parametrize("name", ["decode_int8", "decode_int4"])
def test_quantized_decode_full_size(name):
    """The decode shape (T=64, d=7168, E=128 + 1 shared, k=2, d_ff=2048): routing on every
    token, the output on a seeded sample of tokens (the oracle quantizes each touched expert)."""
    cfg = W.CONFIGS[name]
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    gpu = run_layer(cfg, inp)
    x64, r = oracle_route(cfg, inp)
    rng = np.random.default_rng(cfg.seed)
    tokens = sorted(set(rng.choice(cfg.T, size=10, replace=False).tolist()) | {0, cfg.T - 1})
    rep = check_layer(cfg, inp, gpu, tokens=tokens, x64=x64, r=r)
    print(name, rep)
