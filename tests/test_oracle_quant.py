"""Pins for the oracle's group-wise weight quantization: a hand-worked group (4 and 8 bits),
constant groups, the error bound that follows from the definition, exact round trips of values
already on a group's grid, and the quantized layer equal to the layer on the dequantized
weights."""
import numpy as np
import pytest

import oracle as O
from golden_io import read_kv


def _fixture_group():
    w = (np.arange(128, dtype=np.float64) - 40.0) / 64.0
    return w.reshape(1, 128, 1)


@pytest.mark.parametrize("bits", [4, 8])
def test_quant_fixture_group(bits):
    g = read_kv("quant_group.txt")
    pre = f"b{bits}_"
    q, s, z = O.quantize_groupwise(_fixture_group(), bits)
    assert s.dtype == np.float16 and float(s[0, 0, 0]) == g[pre + "scale"]
    assert int(z[0, 0, 0]) == g[pre + "zero"]
    for k, qk in zip(g[pre + "k"], g[pre + "q"]):
        assert int(q[0, k, 0]) == qk, (bits, k)


def test_quant_constant_groups():
    g = read_kv("quant_group.txt")
    for v, sc, zz, qq in zip(g["const_values"], g["const_scale"], g["const_zero"], g["const_q"]):
        for bits in (4, 8):
            q, s, z = O.quantize_groupwise(np.full((128, 3), v), bits)
            assert float(s[0, 0]) == sc and int(z[0, 0]) == zz and (q == qq).all()
            assert (O.dequantize_groupwise(q, s, z) == v).all()


@pytest.mark.parametrize("bits", [4, 8])
def test_quant_error_bound(bits):
    """|w - w'| <= s/2 where the code is not clamped, and <= (1/2 + (2^b - 1) * 2^-11) * s
    everywhere (the fp16 rounding of s can move the top code off the group's maximum)."""
    rng = np.random.default_rng(bits)
    W = rng.normal(size=(3, 512, 40)) * rng.choice([0.01, 1.0, 30.0], size=(3, 1, 1))
    q, s, z = O.quantize_groupwise(W, bits)
    Wd = O.dequantize_groupwise(q, s, z)
    sg = np.repeat(s.astype(np.float64), 128, axis=-2)
    zg = np.repeat(z.astype(np.float64), 128, axis=-2)
    err = np.abs(W - Wd) / sg
    raw = np.rint(W / sg) + zg
    inside = (raw >= 0) & (raw <= 2 ** bits - 1)
    assert err[inside].max() <= 0.5
    assert err.max() <= 0.5 + (2 ** bits - 1) * 2.0 ** -11
    assert q.max() <= 2 ** bits - 1


@pytest.mark.parametrize("bits", [4, 8])
def test_quant_grid_values_round_trip(bits):
    """Weights that already are (c - z) * s for integer codes c in [0, 2^b - 1] with the group's
    extremes at codes 0 and 2^b - 1 come back exactly."""
    rng = np.random.default_rng(10 + bits)
    top = 2 ** bits - 1
    s = 2.0 ** -7
    z = top // 3
    codes = rng.integers(0, top + 1, size=(128, 7))
    codes[0, :] = 0
    codes[1, :] = top
    W = (codes - z) * s
    q, ss, zz = O.quantize_groupwise(W, bits)
    assert (ss == s).all() and (zz == z).all() and (q == codes).all()
    assert (O.dequantize_groupwise(q, ss, zz) == W).all()


def test_quant_groups_are_independent_along_k():
    """A spike in one group changes only that group's scale and codes."""
    rng = np.random.default_rng(3)
    W = rng.normal(size=(384, 16)) * 0.02
    W2 = W.copy()
    W2[200, 5] = 4.0                         # group 1 (rows 128..255), column 5
    a, b = O.quantize_groupwise(W, 8), O.quantize_groupwise(W2, 8)
    changed = a[1] != b[1]
    assert changed[1, 5] and changed.sum() == 1
    qa, qb = a[0], b[0]
    diff_rows, diff_cols = np.nonzero(qa != qb)
    assert set(diff_cols) == {5} and diff_rows.min() >= 128 and diff_rows.max() < 256


def test_quantized_layer_is_layer_on_dequantized_weights():
    rng = np.random.default_rng(4)
    T, d, E, k, f = 20, 128, 4, 2, 128
    x = rng.normal(size=(T, d))
    Wg = rng.normal(size=(d, E)) / 8
    ex = [tuple(rng.normal(size=sh) / 10 for sh in ((d, f), (d, f), (f, d))) for _ in range(E)]
    deq = []
    for (a, b, c) in ex:
        deq.append(tuple(O.dequantize_groupwise(*O.quantize_groupwise(w, 4)) for w in (a, b, c)))
    out_q = O.layer(x, Wg, k, lambda e: deq[e], E)["out"]
    out_f = O.layer(x, Wg, k, lambda e: ex[e], E)["out"]
    rel = np.linalg.norm(out_q - out_f) / np.linalg.norm(out_f)
    assert 1e-4 < rel < 0.2                   # 4-bit weights move the output, but not wildly
