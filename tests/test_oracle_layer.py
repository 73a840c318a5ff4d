"""Pins for the oracle's experts and whole layer: a hand-worked SwiGLU expert, a dense
every-expert-on-every-token path, the k=E equal-gate reduction to the mean of experts,
linearity of the combine in the gates, and capacity drops."""
import math

import numpy as np
import pytest

import oracle as O
from golden_io import read_kv


def test_swiglu_fixture():
    g = read_kv("swiglu_small.txt")
    ln3 = math.log(3.0)
    x = np.array([[1.0, 2.0]])
    Wg = np.array([[0.0, ln3, 0.0], [0.0, 0.0, -ln3 / 2]])
    Wu = np.array([[5.0, 0.0, 4.0], [0.0, 1.0, 0.0]])
    Wd = np.array([[7.0, 7.0], [1.0, 0.0], [0.0, 1.0]])
    y = O.swiglu_expert(x, Wg, Wu, Wd)
    np.testing.assert_allclose(y[0], g["y"], rtol=0, atol=1e-14)


def test_silu_special_values():
    np.testing.assert_allclose(O.silu([0.0, math.log(3.0), -math.log(3.0)]),
                               [0.0, 0.75 * math.log(3.0), -0.25 * math.log(3.0)], atol=1e-15)
    assert O.silu([-1000.0])[0] == 0.0 and O.silu([1000.0])[0] == 1000.0


def make_layer(rng, T, d, E, f, S=0):
    x = rng.standard_normal((T, d))
    W_g = rng.standard_normal((d, E)) / math.sqrt(d)
    experts = [(rng.standard_normal((d, f)) / math.sqrt(d), rng.standard_normal((d, f)) / math.sqrt(d),
                rng.standard_normal((f, d)) / math.sqrt(f)) for _ in range(E)]
    shared = [(rng.standard_normal((d, f)) / math.sqrt(d), rng.standard_normal((d, f)) / math.sqrt(d),
               rng.standard_normal((f, d)) / math.sqrt(f)) for _ in range(S)]
    return x, W_g, experts, shared


@pytest.mark.parametrize("mode,k,S", [(O.PLAIN, 2, 0), (O.BIAS_SELECT, 3, 2), (O.GUMBEL, 2, 1),
                                      (O.PLAIN, 6, 0)])
def test_routed_layer_equals_dense_layer(mode, k, S):
    rng = np.random.default_rng(11 + k + S)
    T, d, E, f = 24, 12, 6, 10
    x, W_g, experts, shared = make_layer(rng, T, d, E, f, S)
    bias = rng.standard_normal(E)
    u = rng.uniform(2 ** -24, 1 - 2 ** -24, (T, E))
    routed = O.layer(x, W_g, k, lambda e: experts[e], E, mode, bias, u, 0.5, n_shared=S,
                     get_shared=lambda s: shared[s])
    dense = O.layer_dense(x, W_g, k, experts, mode, bias, u, 0.5, shared)
    np.testing.assert_allclose(routed["out"], dense, rtol=0, atol=1e-12)
    # the same layer computed only for a subset of tokens
    toks = [3, 0, 17]
    part = O.layer(x, W_g, k, lambda e: experts[e], E, mode, bias, u, 0.5, n_shared=S,
                   get_shared=lambda s: shared[s], tokens=toks)
    np.testing.assert_allclose(part["out"], dense[toks], rtol=0, atol=1e-12)


def test_k_equals_E_zero_router_is_mean_of_experts():
    """W_g = 0 and bias = 0: every score ties, so with k = E each gate is 1/E and the layer
    output is the plain average of all E experts."""
    rng = np.random.default_rng(5)
    T, d, E, f = 9, 8, 4, 6
    x, _, experts, _ = make_layer(rng, T, d, E, f)
    r = O.layer(x, np.zeros((d, E)), E, lambda e: experts[e], E)
    np.testing.assert_allclose(r["route"]["topk_w"], 1.0 / E, atol=1e-15)
    assert r["route"]["topk_idx"].tolist() == [list(range(E))] * T
    mean = np.zeros((T, d))
    for Wg, Wu, Wd in experts:
        for t in range(T):
            mean[t] += O.swiglu_expert(x[t:t + 1], Wg, Wu, Wd)[0] / E
    np.testing.assert_allclose(r["out"], mean, atol=1e-12)


def test_combine_is_linear_in_gates():
    rng = np.random.default_rng(9)
    T, d, E, f, k = 16, 8, 5, 6, 2
    x, W_g, experts, _ = make_layer(rng, T, d, E, f)
    r = O.route(x, W_g, k)
    a, _ = O.layer_from_routing(x, r["topk_idx"], r["topk_w"], E, None, lambda e: experts[e])
    b, _ = O.layer_from_routing(x, r["topk_idx"], 2.5 * r["topk_w"], E, None, lambda e: experts[e])
    np.testing.assert_allclose(b, 2.5 * a, atol=1e-12)


def test_capacity_drops_zero_the_slot():
    """A dropped slot contributes nothing and the kept gates are not renormalised."""
    rng = np.random.default_rng(2)
    T, d, E, f, k = 10, 6, 3, 4, 1
    x, _, experts, _ = make_layer(rng, T, d, E, f)
    W_g = np.zeros((d, E))
    bias = np.array([1.0, 0.0, 0.0])          # every token picks expert 0
    r = O.layer(x, W_g, k, lambda e: experts[e], E, O.BIAS_SELECT, bias, capacity_override=4)
    assert r["perm"]["n_kept"] == 4
    for t in range(T):
        want = O.swiglu_expert(x[t:t + 1], *experts[0])[0] if t < 4 else np.zeros(d)
        np.testing.assert_allclose(r["out"][t], want, atol=1e-12)


def test_bias_update_hand_values():
    """bias <- 0.99*bias - 0.01*load/mean(load), worked by hand: loads [4,0,2,2] have mean 2."""
    b = np.array([0.5, -0.2, 0.0, 0.1])
    np.testing.assert_allclose(O.bias_update(b, np.array([4, 0, 2, 2])),
                               [0.475, -0.198, -0.01, 0.089], atol=1e-9)
    np.testing.assert_allclose(O.bias_update(np.zeros(2), [3, 1]), [-0.015, -0.005], atol=1e-9)
