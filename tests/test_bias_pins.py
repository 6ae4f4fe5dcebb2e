"""Pins of the oracle's additive score bias (CPU only): reductions to cases
fixed elsewhere (no bias, the causal mask, a per-row shift that softmax
ignores), a closed form (a key-weighted softmax written out by hand),
broadcasting, and finite differences for the backward."""
import numpy as np
import pytest

import oracle


def tiny(B=2, H=2, N=37, d=8, seed=0):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, H, N, d)) for _ in range(4)]


def test_zero_bias_is_no_bias():
    q, k, v, do = tiny()
    z = np.zeros((1, 1, 37, 37))
    o0, l0 = oracle.forward(q, k, v, 0.4, causal=True)
    o1, l1 = oracle.forward(q, k, v, 0.4, causal=True, bias=z)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    for a, b in zip(oracle.backward(q, k, v, do, 0.4, causal=True),
                    oracle.backward(q, k, v, do, 0.4, causal=True, bias=z)):
        assert np.array_equal(a, b)


def test_minus_inf_bias_is_the_causal_mask():
    q, k, v, do = tiny()
    N = q.shape[2]
    i, j = np.indices((N, N))
    bias = np.where(j > i, -np.inf, 0.0)[None, None]
    o0, l0 = oracle.forward(q, k, v, 0.4, causal=True)
    o1, l1 = oracle.forward(q, k, v, 0.4, bias=bias)
    assert np.allclose(o0, o1) and np.allclose(l0, l1)
    for a, b in zip(oracle.backward(q, k, v, do, 0.4, causal=True),
                    oracle.backward(q, k, v, do, 0.4, bias=bias)):
        assert np.allclose(a, b)


def test_row_constant_bias_shifts_lse_only():
    q, k, v, do = tiny()
    B, H, N, _ = q.shape
    c = np.random.default_rng(1).standard_normal((B, H, N, 1)) * 3.0
    bias = np.broadcast_to(c, (B, H, N, N))
    o0, l0 = oracle.forward(q, k, v, 0.4)
    o1, l1 = oracle.forward(q, k, v, 0.4, bias=bias)
    assert np.allclose(o0, o1)
    assert np.allclose(l1, l0 + c[..., 0])
    for a, b in zip(oracle.backward(q, k, v, do, 0.4), oracle.backward(q, k, v, do, 0.4, bias=bias)):
        assert np.allclose(a, b)


def test_log_weights_give_the_weighted_softmax():
    """bias_ij = ln w_j: O_i = sum_j w_j e^{s_ij} v_j / sum_j w_j e^{s_ij},
    evaluated here with explicit loops over one slice."""
    q, k, v, _ = tiny(B=1, H=1, N=9, d=3, seed=2)
    w = np.random.default_rng(3).uniform(0.1, 4.0, 9)
    bias = np.broadcast_to(np.log(w)[None, :], (9, 9))[None, None]
    o, lse = oracle.forward(q, k, v, 0.7, bias=bias)
    for i in range(9):
        num = np.zeros(3)
        den = 0.0
        for jj in range(9):
            e = w[jj] * np.exp(0.7 * float(np.dot(q[0, 0, i], k[0, 0, jj])))
            num += e * v[0, 0, jj]
            den += e
        assert np.allclose(o[0, 0, i], num / den)
        assert np.isclose(lse[0, 0, i], np.log(den))


def test_broadcast_equals_tiled():
    q, k, v, do = tiny()
    B, H, N, _ = q.shape
    one = np.random.default_rng(4).standard_normal((1, 1, N, N))
    per_head = np.random.default_rng(5).standard_normal((1, H, N, N))
    for bias in (one, per_head):
        tiled = np.broadcast_to(bias, (B, H, N, N)).copy()
        a = oracle.forward(q, k, v, 0.4, bias=bias)
        b = oracle.forward(q, k, v, 0.4, bias=tiled)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_with_bias_matches_finite_differences(causal):
    q, k, v, do = tiny(B=1, H=1, N=10, d=4, seed=6)
    bias = np.random.default_rng(7).standard_normal((1, 1, 10, 10))
    dq, dk, dv, _ = oracle.backward(q, k, v, do, 0.6, causal=causal, bias=bias)

    def loss(q_, k_, v_):
        o, _ = oracle.forward(q_, k_, v_, 0.6, causal=causal, bias=bias)
        return float(np.sum(o * do))

    eps = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            ap, am = [q, k, v], [q, k, v]
            ap[which], am[which] = xp, xm
            num[idx] = (loss(*ap) - loss(*am)) / (2 * eps)
        assert np.max(np.abs(num - g)) < 1e-6 * max(1.0, np.max(np.abs(g)))


def test_sampled_rows_with_bias():
    q, k, v, do = tiny(B=2, H=2, N=300, d=8, seed=8)
    bias = np.random.default_rng(9).standard_normal((2, 1, 300, 300))
    o, lse = oracle.forward(q, k, v, 0.4, causal=True, bias=bias)
    dq, dk, dv, dd = oracle.backward(q, k, v, do, 0.4, causal=True, bias=bias)
    rows = np.stack([np.stack([np.array([0, 7, 128, 299])] * 2)] * 2)
    ro, rl = oracle.forward_rows(q, k, v, 0.4, rows, causal=True, bias=bias)
    assert np.allclose(ro, np.take_along_axis(o, rows[..., None], 2))
    rdq = oracle.backward_query_rows(q, k, v, do, 0.4, rows, causal=True, bias=bias)
    assert np.allclose(rdq, np.take_along_axis(dq, rows[..., None], 2))
    lse_all, d_all = oracle.row_stats(q, k, v, do, 0.4, causal=True, bias=bias)
    assert np.allclose(lse_all, lse) and np.allclose(d_all, dd)
    rdk, rdv = oracle.backward_key_rows(q, k, v, do, 0.4, rows, lse_all, d_all, causal=True,
                                        bias=bias)
    assert np.allclose(rdk, np.take_along_axis(dk, rows[..., None], 2))
    assert np.allclose(rdv, np.take_along_axis(dv, rows[..., None], 2))
