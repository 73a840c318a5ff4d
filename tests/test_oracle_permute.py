"""Pins for the oracle's dispatch: a hand-worked fixture, the capacity formula's own cases, a
second independent construction (stable sort), and the invariants every dispatch must keep."""
import numpy as np
import pytest

import oracle as O
from golden_io import read_kv, read_rows


def test_permute_fixture():
    g = read_kv("permute_small.txt")
    idx = np.array(g["topk_idx"]).reshape(g["T"], g["k"])
    for fn in (O.permute, O.permute_by_sort):
        p = fn(idx, g["E"], g["C"])
        assert p["counts"].tolist() == g["counts"]
        assert p["offsets"].tolist() == g["offsets"]
        assert p["perm_slot"].tolist() == g["perm_slot"]
        assert p["slot_pos"].tolist() == g["slot_pos"]


def test_capacity_fixture():
    for T, k, E, cf, ov, want in read_rows("capacity.txt"):
        c = O.capacity(int(T), int(k), int(E), float(cf), int(ov))
        assert (c if c is not None else -1) == int(want), (T, k, E, cf, ov)


def random_idx(rng, T, E, k, skew=None):
    idx = np.empty((T, k), dtype=np.int64)
    p = None
    if skew is not None:
        p = np.arange(1, E + 1, dtype=float) ** -skew
        p /= p.sum()
    for t in range(T):
        idx[t] = rng.choice(E, size=k, replace=False, p=p)
    return idx


def check_invariants(idx, E, C, p):
    T, k = idx.shape
    counts, offsets = p["counts"], p["offsets"]
    perm_slot, slot_pos = p["perm_slot"], p["slot_pos"]
    assert counts.sum() == T * k
    kept = counts if C is None else np.minimum(counts, C)
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), kept)
    n = offsets[E]
    assert n == p["n_kept"] and n == (slot_pos >= 0).sum()
    assert np.all(perm_slot[n:] == -1)
    for pos in range(n):                        # inverse maps on kept slots
        assert slot_pos[perm_slot[pos]] == pos
    for e in range(E):                          # one expert per segment, tokens increasing
        seg = perm_slot[offsets[e]:offsets[e + 1]]
        assert np.all(idx.reshape(-1)[seg] == e)
        assert np.all(np.diff(seg // k) > 0)
    if C is not None:                           # the dropped slots are each expert's latest
        for e in range(E):
            slots = np.nonzero(idx.reshape(-1) == e)[0]
            assert np.all(slot_pos[slots[:C]] >= 0) and np.all(slot_pos[slots[C:]] == -1)


@pytest.mark.parametrize("T,E,k,C,skew", [
    (1, 1, 1, None, None), (7, 4, 2, None, None), (64, 8, 2, 1, None), (64, 8, 3, 5, 1.5),
    (100, 16, 4, None, 2.0), (50, 6, 6, 10, None), (33, 5, 1, 1000, None), (128, 32, 8, 3, 1.1)])
def test_permute_two_constructions_agree(T, E, k, C, skew):
    rng = np.random.default_rng(T * 31 + E)
    idx = random_idx(rng, T, E, k, skew)
    a = O.permute(idx, E, C)
    b = O.permute_by_sort(idx, E, C)
    for key in ("counts", "offsets", "perm_slot", "slot_pos"):
        assert np.array_equal(a[key], b[key]), key
    check_invariants(idx, E, C, a)


def test_all_tokens_to_one_expert():
    T, k, E = 20, 1, 4
    idx = np.zeros((T, k), dtype=np.int64)
    p = O.permute(idx, E, 3)
    assert p["counts"].tolist() == [20, 0, 0, 0]
    assert p["offsets"].tolist() == [0, 3, 3, 3, 3]
    assert p["perm_slot"][:3].tolist() == [0, 1, 2]
    assert (p["slot_pos"] >= 0).sum() == 3


def test_capacity_at_least_all_slots_drops_nothing():
    rng = np.random.default_rng(1)
    idx = random_idx(rng, 40, 8, 3)
    a = O.permute(idx, 8, 40 * 3)
    b = O.permute(idx, 8, None)
    assert np.array_equal(a["slot_pos"], b["slot_pos"])
    assert a["n_kept"] == 120
