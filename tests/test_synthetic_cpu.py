"""The seeded input generators follow the stated recipe: 1% outlier channels
scaled x20, the stated distributions and draw order, the workload shapes, and
the stack's chaining of output columns into the next linear's input."""
import numpy as np
import pytest

import synthetic as sy


def _f(bits):
    return bits.view(np.float16).astype(np.float64)


@pytest.mark.parametrize("K,n", [(1024, 10), (2048, 20), (3072, 31), (4096, 41), (14336, 143), (64, 1)])
def test_outlier_channel_counts(K, n):
    assert sy.n_outlier_channels(K) == n


def test_activation_distribution_and_outliers():
    X, idx = sy.make_activations(np.random.default_rng(3), 4096, 1024)
    assert X.dtype == np.uint16 and X.shape == (4096, 1024)
    assert len(idx) == 10 and len(set(idx.tolist())) == 10 and np.all(np.diff(idx) > 0)
    x = _f(X)
    out = np.zeros(1024, bool)
    out[idx] = True
    std = x.std(axis=0)
    assert np.all(np.abs(std[~out] - 1.0) < 0.06)        # N(0, 1)
    assert np.all(np.abs(std[out] - 20.0) < 20 * 0.06)   # the same draws x 20
    assert abs(x[:, ~out].mean()) < 0.01


def test_linear_case_distributions_and_determinism():
    c = sy.make_linear_case(512, 1024, 2048, 32, seed=7)
    assert c.W.dtype == np.float32 and c.W.shape == (2048, 1024)
    assert abs(c.W.std() - 0.02) < 0.0005 and abs(c.W.mean()) < 0.0002
    for L, shape in ((c.L_down, (1024, 32)), (c.L_up, (32, 2048))):
        assert L.shape == shape and abs(_f(L).std() - 0.02) < 0.001
    cs = _f(c.colscale)
    assert cs.min() >= 0.5 and cs.max() <= 1.5 and abs(cs.mean() - 1.0) < 0.03
    assert abs(_f(c.bias).std() - 0.1) < 0.01
    d = sy.make_linear_case(512, 1024, 2048, 32, seed=7)
    for a, b in ((c.X, d.X), (c.W, d.W), (c.L_down, d.L_down), (c.L_up, d.L_up), (c.colscale, d.colscale),
                 (c.bias, d.bias)):
        assert np.array_equal(a, b)
    e = sy.make_linear_case(512, 1024, 2048, 32, seed=8)
    assert not np.array_equal(c.W, e.W) and not np.array_equal(c.X, e.X)


def test_draw_order_x_first():
    # X is drawn first, so the X of a case depends on its seed and shape only, not on N or r
    a = sy.make_linear_case(64, 1024, 1024, 32, seed=0)
    b = sy.make_linear_case(64, 1024, 4096, 16, seed=0)
    assert np.array_equal(a.X, b.X) and np.array_equal(a.outliers, b.outliers)


def test_workload_shapes():
    assert sy.SINGLE_LINEAR == dict(M=64, K=1024, N=1024, r=32)
    assert {k: (v["K"], v["N"]) for k, v in sy.DECODER_LAYER_M700.items()} == {
        "qkv": (1024, 4096), "o": (2048, 1024), "gate_up": (1024, 6144), "down": (3072, 1024)}
    assert all(v["M"] == 700 and v["r"] == 32 for v in sy.DECODER_LAYER_M700.values())
    assert [s["M"] for s in sy.SMALL_M_SWEEP] == [1, 4, 16, 32, 76]
    assert all((s["K"], s["N"]) == (4096, 4096) for s in sy.SMALL_M_SWEEP)
    assert {k: (v["M"], v["K"], v["N"]) for k, v in sy.PREFILL.items()} == {
        "gate_up_style": (8192, 4096, 14336), "down_style": (8192, 14336, 4096)}


def test_stack_chaining_and_seeding():
    assert sy.STACK_LAYERS == 28
    # each linear's output feeds the next linear's K columns, wrapping into the next layer
    for j, (_, K, N) in enumerate(sy.STACK_LINEARS):
        assert sy.stack_next_k(j) <= N
    assert [sy.stack_next_k(j) for j in range(4)] == [2048, 1024, 3072, 1024]
    a, b, c = sy.make_stack_linear(0, 1), sy.make_stack_linear(0, 1), sy.make_stack_linear(1, 1)
    assert (a.name, a.K, a.N) == ("o", 2048, 1024)
    assert np.array_equal(a.W, b.W) and not np.array_equal(a.W, c.W)
    assert sy.make_stack_input(700).shape == (700, 1024)
