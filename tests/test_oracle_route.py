"""Pins for the oracle's router: top-k by brute force, gates by closed form, Gumbel noise by its
inverse, and hand-worked fixtures."""
import itertools
import math

import numpy as np
import pytest

import oracle as O
from golden_io import read_kv


def brute_topk(s_row, k):
    """The unique k-subset that beats every outside expert under (score desc, index asc),
    listed in that order; found by enumerating every subset."""
    E = len(s_row)
    before = lambda a, b: s_row[a] > s_row[b] or (s_row[a] == s_row[b] and a < b)
    winners = []
    for sub in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in sub]
        if all(before(a, b) for a in sub for b in rest):
            winners.append(sub)
    assert len(winners) == 1
    chosen = list(winners[0])
    # order inside the set by pairwise comparisons (selection, not a library sort)
    ordered = []
    while chosen:
        best = chosen[0]
        for c in chosen[1:]:
            if before(c, best):
                best = c
        ordered.append(best)
        chosen.remove(best)
    return ordered


@pytest.mark.parametrize("E", [1, 2, 3, 4])
def test_topk_bruteforce_small(E):
    rng = np.random.default_rng(E)
    for trial in range(40):
        T = int(rng.integers(1, 9))
        # small integer scores force many exact ties
        s = rng.integers(-2, 3, size=(T, E)).astype(np.float64)
        for k in range(1, E + 1):
            got = O.topk(s, k)
            for t in range(T):
                assert list(got[t]) == brute_topk(list(s[t]), k)


def test_topk_bruteforce_continuous():
    rng = np.random.default_rng(7)
    for _ in range(50):
        s = rng.standard_normal((8, 4))
        for k in range(1, 5):
            got = O.topk(s, k)
            for t in range(8):
                assert list(got[t]) == brute_topk(list(s[t]), k)


def test_route_gates_fixture():
    g = read_kv("gates_small.txt")
    # case A: plain
    logits = np.array([[0.0, math.log(3.0), -5.0]])
    s = O.selection_scores(logits, O.PLAIN)
    idx = O.topk(s, 2)
    w = O.gates(logits, s, idx, O.PLAIN)
    assert list(idx[0]) == g["A_idx"]
    np.testing.assert_allclose(w[0], g["A_w"], rtol=0, atol=1e-15)
    # case B: bias enters selection only
    logits = np.array([[1.0, 0.9, 0.0]])
    s = O.selection_scores(logits, O.BIAS_SELECT, expert_bias=np.array([0.0, 0.0, 2.0]))
    idx = O.topk(s, 2)
    w = O.gates(logits, s, idx, O.BIAS_SELECT)
    assert list(idx[0]) == g["B_idx"]
    np.testing.assert_allclose(w[0], g["B_w"], rtol=0, atol=1e-15)
    # case C: exact ties go to the lower index
    logits = np.array([[0.5, 0.5, 0.5, 0.1]])
    s = O.selection_scores(logits, O.PLAIN)
    idx = O.topk(s, 2)
    assert list(idx[0]) == g["C_idx"]
    np.testing.assert_allclose(O.gates(logits, s, idx, O.PLAIN)[0], g["C_w"], atol=1e-15)


def test_route_end_to_end_linear_layer():
    """route() = linear layer without bias: an identity input row returns W_g's rows as logits."""
    W_g = np.array([[0.0, 2.0, 1.0], [3.0, -1.0, 0.5]])
    x = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    r = O.route(x, W_g, 2)
    np.testing.assert_array_equal(r["logits"], [[0, 2, 1], [3, -1, 0.5], [3, 1, 1.5]])
    assert r["topk_idx"].tolist() == [[1, 2], [0, 2], [0, 2]]


def test_gates_sum_to_one_and_order():
    rng = np.random.default_rng(3)
    for mode in (O.PLAIN, O.BIAS_SELECT, O.GUMBEL):
        x = rng.standard_normal((50, 16))
        W_g = rng.standard_normal((16, 12)) / 4
        bias = rng.standard_normal(12)
        u = rng.uniform(2 ** -24, 1 - 2 ** -24, size=(50, 12))
        r = O.route(x, W_g, 4, mode, bias, u, 0.5)
        np.testing.assert_allclose(r["topk_w"].sum(1), 1.0, atol=1e-14)
        sel = np.take_along_axis(r["scores"], r["topk_idx"].astype(np.int64), 1)
        assert np.all(np.diff(sel, axis=1) <= 0)             # descending scores
        if mode != O.BIAS_SELECT:
            assert np.all(np.diff(r["topk_w"], axis=1) <= 1e-15)  # gates follow the ranking


def test_gumbel_noise_inverse():
    """u = exp(-exp(-a)) is the Gumbel CDF at a, so g(u) = -log(-log u) must return a."""
    a = np.linspace(-2.5, 6.0, 200)
    u = np.exp(-np.exp(-a))
    np.testing.assert_allclose(O.gumbel_noise(u), a, rtol=0, atol=1e-9)


def test_gumbel_scores_temperature():
    """score = (logit + g) / tau: with g known, the score is an affine map of the logits."""
    a = np.array([[0.3, -1.0, 2.0]])
    u = np.exp(-np.exp(-a))
    logits = np.array([[1.0, 0.5, -0.25]])
    s = O.selection_scores(logits, O.GUMBEL, gumbel_u=u, tau=0.5)
    np.testing.assert_allclose(s, (logits + a) * 2.0, atol=1e-9)
    idx = O.topk(s, 2)
    assert idx.tolist() == [[2, 0]]
    w = O.gates(logits, s, idx, O.GUMBEL)
    # GUMBEL gates: softmax over the selected perturbed scores s = [3.5, 2.6]
    e = math.exp(3.5 - 2.6)
    np.testing.assert_allclose(w[0], [e / (1 + e), 1 / (1 + e)], atol=1e-9)


def test_tie_margin():
    s = np.array([[3.0, 1.0, 2.0, 2.0 + 4e-6], [5.0, 0.0, 1.0, 3.0]])
    m = O.tie_margin(s, 2)
    np.testing.assert_allclose(m, [4e-6, 2.0])
    assert O.tie_margin(s, 4)[1] == 1.0   # k = E: gaps among all E scores


def test_bf16_widening_roundtrip():
    vals = np.array([0.0, 1.0, -2.5, 3.140625, 1e-3, -65280.0])
    bits = O.f64_to_bf16_bits(vals)
    back = O.bf16_bits_to_f64(bits)
    np.testing.assert_allclose(back, vals, rtol=2 ** -8)
    assert O.f64_to_bf16_bits([1.0])[0] == 0x3F80
    assert O.f64_to_bf16_bits([1.0 + 2 ** -8])[0] == 0x3F80     # tie -> even
    assert O.f64_to_bf16_bits([1.0 + 3 * 2 ** -8])[0] == 0x3F82


def brute_group_topk(s_row, k, n_groups, g):
    """Group-limited top-k by enumeration of group subsets (definition, no sorting)."""
    E = len(s_row)
    size = E // n_groups
    gs = [max(s_row[i * size:(i + 1) * size]) for i in range(n_groups)]
    before_g = lambda a, b: gs[a] > gs[b] or (gs[a] == gs[b] and a < b)
    chosen = None
    for sub in itertools.combinations(range(n_groups), g):
        rest = [x for x in range(n_groups) if x not in sub]
        if all(before_g(a, b) for a in sub for b in rest):
            chosen = sub
    allowed = [e for e in range(E) if e // size in chosen]
    masked = [s_row[e] if e in allowed else -math.inf for e in range(E)]
    return brute_topk(masked, k)


def brute_group_margin(s_row, n_groups, g):
    """The group decision's gap by enumeration: over every way of keeping g groups such that no
    dropped group scores above a kept one, the weakest kept group score minus the strongest
    dropped one (inf when every group is kept)."""
    if g >= n_groups:
        return math.inf
    size = len(s_row) // n_groups
    gs = [max(s_row[i * size:(i + 1) * size]) for i in range(n_groups)]
    gaps = []
    for sub in itertools.combinations(range(n_groups), g):
        rest = [x for x in range(n_groups) if x not in sub]
        lo, hi = min(gs[a] for a in sub), max(gs[b] for b in rest)
        if lo >= hi:
            gaps.append(lo - hi)
    return max(gaps)


def test_group_limited_fixture():
    from golden_io import read_kv
    g = read_kv("group_limited.txt")
    s = np.array([[0.9, 0.1, 0.8, 0.85, 0.3, 0.2, 0.95, -1.0]])
    for gk, key in ((1, "g1"), (2, "g2"), (3, "g3")):
        assert O.topk(O.group_limit(s, 4, gk), 2)[0].tolist() == g[key]
    s2 = np.array([[0.5, 0.0, 0.5, 0.4, 0.1, 0.1, 0.2, 0.2]])
    assert O.topk(O.group_limit(s2, 4, 1), 2)[0].tolist() == g["tie1"]


def test_group_margin_fixture():
    """The group decision's gap, worked by hand: the gaps between adjacent sorted group scores
    all differ, so indexing the wrong pair, or scoring a group by a member other than its
    largest, fails."""
    from golden_io import read_kv
    g = read_kv("group_limited.txt")
    s3 = np.array([[0.7, -0.2, 0.1, 0.65, 1.0, 0.3, -0.5, 0.4]])
    for gk, key in ((1, "m1"), (2, "m2"), (3, "m3")):
        np.testing.assert_allclose(O.group_margin(s3, 4, gk), [g[key]], rtol=0, atol=1e-12)
    s2 = np.array([[0.5, 0.0, 0.5, 0.4, 0.1, 0.1, 0.2, 0.2]])
    np.testing.assert_allclose(O.group_margin(s2, 4, 1), [g["mtie1"]], rtol=0, atol=1e-12)
    np.testing.assert_allclose(O.group_margin(s2, 4, 2), [g["mtie2"]], rtol=0, atol=1e-12)


def test_group_limited_bruteforce():
    rng = np.random.default_rng(17)
    for _ in range(60):
        n_groups = int(rng.choice([2, 3, 4]))
        size = int(rng.integers(1, 4))
        E = n_groups * size
        g = int(rng.integers(1, n_groups + 1))
        k = int(rng.integers(1, g * size + 1))
        s = rng.integers(-2, 3, size=(5, E)).astype(np.float64)
        got = O.topk(O.group_limit(s, n_groups, g), k)
        marg = O.group_margin(s, n_groups, g)
        for t in range(5):
            assert list(got[t]) == brute_group_topk(list(s[t]), k, n_groups, g)
            assert marg[t] == brute_group_margin(list(s[t]), n_groups, g)


def test_group_limited_all_groups_is_plain_topk():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((30, 12))
    assert np.array_equal(O.topk(O.group_limit(s, 4, 4), 3), O.topk(s, 3))
    np.testing.assert_array_equal(O.group_margin(s, 4, 4), np.inf)
