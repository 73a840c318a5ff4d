"""The four large workloads at full size, in the launch configuration the benchmark times:
routing bit-exact on every token (near-ties exempt and counted), dispatch bit-exact on every
slot, and the layer output against the oracle on every token (fine-grained prefill, decode) or,
for the two layers whose full fp64 evaluation takes minutes, on every row tile: the tokens at the
first and last position of every 128-row block of every expert's segment (so both CTAs of every
256-row CTA-pair tile, and every 128-row tile, contribute checked rows), the first and last
token, and a few tokens with dropped slots."""
import numpy as np
import pytest
import torch

import workloads as W
from moe_harness import run_layer, check_layer, to_device, oracle_route

pytestmark = pytest.mark.gpu


def tile_tokens(offsets, perm_slot, k, block=128):
    """Tokens whose slots sit at the first and last position of every `block`-row block of every
    expert's segment of the expert-ordered rows (the GPU's own dispatch)."""
    toks = set()
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for p0 in range(lo, hi, block):
            for p in (p0, min(p0 + block, hi) - 1):
                toks.add(int(perm_slot[p]) // k)
    return toks


@pytest.mark.parametrize("name", ["fine_grained", "decode", "skewed_cap", "gumbel"])
def test_full_size_workload(name):
    cfg = W.CONFIGS[name]
    inp = to_device(W.make_inputs(cfg, weights_device="cuda"))
    gpu = run_layer(cfg, inp)
    x64, r = oracle_route(cfg, inp)
    if name in ("fine_grained", "decode"):
        tokens = None                      # every output element
    else:
        toks = tile_tokens(gpu["offsets"], gpu["perm_slot"], cfg.k) | {0, cfg.T - 1}
        if name == "skewed_cap":
            dropped = np.nonzero((gpu["slot_pos"].reshape(cfg.T, cfg.k) < 0).any(1))[0]
            toks |= set(dropped[:4].tolist())
        tokens = sorted(toks)
    rep = check_layer(cfg, inp, gpu, tokens=tokens, x64=x64, r=r)
    print(name, rep, "checked tokens:", cfg.T if tokens is None else len(tokens))
    if tokens is not None:
        # every 128-row block of the expert-ordered rows holds a checked token's slot
        slot_tok = gpu["perm_slot"][: int(gpu["offsets"][-1])] // cfg.k
        checked = np.isin(slot_tok, np.array(tokens))
        n_blocks = 0
        for e in range(cfg.E):
            lo, hi = int(gpu["offsets"][e]), int(gpu["offsets"][e + 1])
            for p0 in range(lo, hi, 128):
                n_blocks += 1
                assert checked[p0:min(p0 + 128, hi)].any(), (e, p0)
        assert n_blocks >= cfg.E // 2
    if name == "skewed_cap":
        assert rep["C"] == 320 and rep["n_kept"] < cfg.T * cfg.k
        fully = np.nonzero((gpu["slot_pos"].reshape(cfg.T, cfg.k) < 0).all(1))[0]
        if fully.size:
            assert torch.count_nonzero(gpu["out_t"][torch.as_tensor(fully[:64])]) == 0
    if name == "decode":
        hit = np.unique(gpu["topk_idx"]).size
        assert 60 <= hit <= 100
