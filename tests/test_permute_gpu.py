"""Dispatch kernels (moe_permute) bit-exact against the oracle dispatch on the same indices."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_moe_layer_route_gb300 as M

pytestmark = pytest.mark.gpu


def gpu_permute(idx, E, C_override=0, capacity_factor=0.0):
    T, k = idx.shape
    mc = M.MoeConfig.make(T, 64, E, k, 64, capacity_factor=capacity_factor,
                          capacity_override=C_override)
    dev = "cuda"
    ti = torch.as_tensor(idx.astype(np.int32), device=dev)
    counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    perm_slot = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    slot_pos = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    ws = M.alloc_workspace(mc)
    M.permute(mc, ti, counts, offsets, perm_slot, slot_pos, ws)
    status = M.device_status(ws)
    return {"counts": counts.cpu().numpy(), "offsets": offsets.cpu().numpy(),
            "perm_slot": perm_slot.cpu().numpy(), "slot_pos": slot_pos.cpu().numpy(),
            "status": status}


def random_idx(rng, T, E, k, skew=None):
    if skew is None:
        keys = rng.random((T, E))
    else:
        keys = rng.random((T, E)) * (np.arange(1, E + 1) ** -skew)[None, :]
    return np.argsort(-keys, axis=1)[:, :k]


@pytest.mark.parametrize("T,E,k,C,skew", [
    (1, 1, 1, 0, None), (5, 3, 2, 1, None), (300, 8, 2, 0, None), (300, 8, 2, 40, 1.0),
    (1024, 64, 6, 0, None), (1025, 64, 6, 100, 1.2), (4096, 128, 2, 1, 2.0),
    (16384, 128, 2, 320, 1.5), (3000, 256, 8, 0, None), (999, 17, 3, 177, 0.5),
    (64, 128, 2, 0, None), (50, 4, 4, 50 * 4, None)])
def test_permute_matches_oracle(T, E, k, C, skew):
    rng = np.random.default_rng(T * 7 + E)
    idx = random_idx(rng, T, E, k, skew)
    g = gpu_permute(idx, E, C)
    p = O.permute(idx, E, C if C > 0 else None)
    assert g["status"] == 0
    for key in ("counts", "offsets", "perm_slot", "slot_pos"):
        assert np.array_equal(g[key], p[key]), key


def test_permute_capacity_factor_matches_exact_formula():
    rng = np.random.default_rng(5)
    T, E, k = 4096, 64, 6
    idx = random_idx(rng, T, E, k, 1.3)
    for cf in (1.0, 1.1, 1.25, 2.0, 0.01):
        g = gpu_permute(idx, E, 0, cf)
        p = O.permute(idx, E, O.capacity(T, k, E, cf))
        assert np.array_equal(g["slot_pos"], p["slot_pos"]), cf
        assert np.array_equal(g["offsets"], p["offsets"]), cf


def test_permute_all_to_one_expert():
    idx = np.zeros((5000, 1), dtype=np.int64)
    g = gpu_permute(idx, 8, 1234)
    p = O.permute(idx, 8, 1234)
    for key in ("counts", "offsets", "perm_slot", "slot_pos"):
        assert np.array_equal(g[key], p[key]), key


def test_permute_bad_index_reported_not_faulted():
    rng = np.random.default_rng(1)
    idx = random_idx(rng, 200, 8, 2)
    idx[17, 1] = 8          # out of range
    idx[150, 0] = -3
    g = gpu_permute(idx, 8)
    assert g["status"] & M.DEVFAULT_BAD_EXPERT_INDEX
    assert g["slot_pos"][17 * 2 + 1] == -1 and g["slot_pos"][300] == -1
    good = np.ones(400, bool)
    good[[35, 300]] = False
    assert g["counts"].sum() == 398 and (g["slot_pos"][good] >= 0).all()
