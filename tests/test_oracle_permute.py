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


# ---------------------------------------------------------------------------- Level-2 re-route
def _level1(s, k, E, C):
    idx = O.topk(s, k)
    return idx, O.permute(idx, E, C)["slot_pos"]


def test_reroute_fixture_single_slot():
    g = read_kv("reroute_small.txt")
    s = np.array(g["a_scores"], float).reshape(5, 3)
    idx, sp = _level1(s, 1, 3, 2)
    rr = O.overflow_reroute(idx, sp, s, 3, 2)
    assert rr["topk_idx"][:, 0].tolist() == g["a_final"]
    p = O.permute(rr["topk_idx"], 3, 2)
    assert p["offsets"].tolist() == g["a_offsets"]
    assert p["perm_slot"].tolist() == g["a_perm_slot"]
    assert (p["slot_pos"] >= 0).all()
    assert rr["margin"].tolist() == g["a_margin"]


def test_reroute_fixture_token_keeps_distinct_experts():
    g = read_kv("reroute_small.txt")
    s = np.array(g["b_scores"], float).reshape(3, 4)
    idx, sp = _level1(s, 2, 4, 2)
    assert sp.tolist() == [0, 2, 1, 3, -1, 4]
    rr = O.overflow_reroute(idx, sp, s, 4, 2)
    assert rr["topk_idx"].reshape(-1).tolist() == g["b_final"]
    w = O.gates(s, s, rr["topk_idx"], O.PLAIN)
    np.testing.assert_allclose(w[2], g["b_t2_gates"], rtol=0, atol=1e-15)


def _random_case(rng, T, E, k, C, integer):
    s = rng.integers(0, 4, (T, E)).astype(float) if integer else rng.normal(size=(T, E))
    s += np.log(np.arange(1, E + 1))[rng.permutation(E)] * -1.5   # skewed, so slots overflow
    return s


@pytest.mark.parametrize("seed", range(12))
def test_reroute_walk_equals_proposals(seed):
    rng = np.random.default_rng(seed)
    T, E = int(rng.integers(5, 60)), int(rng.integers(2, 12))
    k = int(rng.integers(1, min(E, 4) + 1))
    C = int(rng.integers(1, max(2, T * k // E) + 1))
    s = _random_case(rng, T, E, k, C, integer=seed % 2 == 0)
    idx, sp = _level1(s, k, E, C)
    a = O.overflow_reroute(idx, sp, s, E, C)["topk_idx"]
    b = O.overflow_reroute_by_proposals(idx, sp, s, E, C)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("seed", range(8))
def test_reroute_invariants(seed):
    """Checked on the final assignment alone: capacity, distinct experts per token, and that no
    re-routed slot passed over an expert it prefers that still had room at its turn."""
    rng = np.random.default_rng(100 + seed)
    T, E, k = 80, 8, 2
    C = int(rng.integers(4, 22))
    s = _random_case(rng, T, E, k, C, integer=seed % 2 == 1)
    idx, sp = _level1(s, k, E, C)
    rr = O.overflow_reroute(idx, sp, s, E, C)
    fin, rer = rr["topk_idx"], rr["rerouted"]
    dropped1 = (sp < 0).reshape(T, k)
    assert not (rer & ~dropped1).any()                       # only dropped slots move
    assert np.array_equal(fin[~rer], idx[~rer])
    p = O.permute(fin, E, C)
    live = (p["slot_pos"] >= 0).reshape(T, k)
    assert np.array_equal(live, ~dropped1 | rer)             # every re-routed slot is kept
    for t in range(T):
        es = fin[t][live[t]]
        assert len(set(es.tolist())) == len(es)
    kept1 = np.bincount(idx[~dropped1], minlength=E)
    for t in range(T):
        for j in np.nonzero(rer[t])[0]:
            e = fin[t, j]
            # load of each expert when (t, j) took its turn: Level-1 slots + earlier re-routes
            before = kept1.copy()
            for (tt, jj) in zip(*np.nonzero(rer)):
                if (tt, jj) < (t, j):
                    before[fin[tt, jj]] += 1
            mine = set(fin[t][live[t]].tolist()) - {e}
            for e2 in range(E):
                better = s[t, e2] > s[t, e] or (s[t, e2] == s[t, e] and e2 < e)
                if better and e2 not in mine:
                    assert before[e2] >= C, (t, j, e, e2)


def test_reroute_without_overflow_is_identity():
    rng = np.random.default_rng(5)
    s = rng.normal(size=(40, 6))
    idx, sp = _level1(s, 2, 6, 40)
    rr = O.overflow_reroute(idx, sp, s, 6, 40)
    assert np.array_equal(rr["topk_idx"], idx) and not rr["rerouted"].any()


def test_reroute_layer_reduces_to_level1_when_nothing_overflows():
    rng = np.random.default_rng(9)
    T, d, E, k, f = 24, 16, 4, 2, 8
    x = rng.normal(size=(T, d))
    Wg = rng.normal(size=(d, E)) / 4
    ex = [tuple(rng.normal(size=sh) / 4 for sh in ((d, f), (d, f), (f, d))) for _ in range(E)]
    a = O.layer(x, Wg, k, lambda e: ex[e], E, capacity_override=T * k, reroute=True)
    b = O.layer(x, Wg, k, lambda e: ex[e], E, capacity_override=T * k)
    np.testing.assert_array_equal(a["out"], b["out"])
    Wg2 = Wg.copy()
    Wg2[:, 0] += 1.0                                     # every token now prefers experts 0, 1
    Wg2[:, 1] += 0.9
    x2 = x + 1.0
    c = O.layer(x2, Wg2, k, lambda e: ex[e], E, capacity_override=4, reroute=True)
    c1 = O.layer(x2, Wg2, k, lambda e: ex[e], E, capacity_override=4)
    assert c1["perm"]["n_kept"] < E * 4                  # Level 1 leaves room unused ...
    assert c["perm"]["n_kept"] == E * 4                  # ... that Level 2 fills (16 < T*k = 48)
