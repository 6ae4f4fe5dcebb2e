"""Pins of the oracle's dropout (CPU only), against what fixes it from
outside: the published known-answer values of Philox4x32-10, the counter
layout evaluated element by element with the scalar generator, the keep
statistics, the reduction to plain attention at p = 0, the expectation over
seeds, and finite differences of the oracle's own forward for the backward."""
import numpy as np
import pytest

import oracle
from oracle import dropout as D


# Known-answer values of Philox4x32-10 distributed with the generator's
# reference implementation (Random123, by the authors of "Parallel random
# numbers: as easy as 1, 2, 3"): (counter, key) -> output.
KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", KAT)
def test_philox_known_answers(ctr, key, want):
    assert D.philox4x32_10_scalar(ctr, key) == want
    got = D.philox4x32_10(*[np.array([c]) for c in ctr], *key)
    assert tuple(int(w[0]) for w in got) == want


def test_keep_mask_layout_element_by_element():
    """Every sampled element (i, j) of head bh equals the stated rule applied
    to one scalar Philox call: counter (j//8, i, bh, offset), key (seed lo,
    seed hi), half j%2 of word (j%8)//2, kept iff >= t."""
    rng = np.random.default_rng(3)
    seed, offset, bh, p = 0x0123456789ABCDEF, 41, 5, 0.3
    rows = rng.integers(0, 5000, 40)
    cols = rng.integers(0, 5000, 50)
    z = D.keep_mask(rows, cols, bh, p, seed, offset)
    t = D.threshold(p)
    for a, i in enumerate(rows):
        for c, j in enumerate(cols):
            w = D.philox4x32_10_scalar((j // 8, i, bh, offset),
                                       (seed & 0xFFFFFFFF, seed >> 32))
            u = (w[(j % 8) // 2] >> (16 * (j % 2))) & 0xFFFF
            assert z[a, c] == (u >= t)


def test_threshold_and_scale():
    assert D.threshold(0.0) == 0 and D.keep_scale(0.0) == 1.0
    assert D.threshold(0.5) == 32768 and D.keep_scale(0.5) == 2.0
    assert D.threshold(0.1) == 6554          # 6553.6 rounded
    assert D.threshold(0.99999) == 65535
    assert D.threshold(0.9999999) == 65535   # 65535.99 rounds to 65536: clamped
    with pytest.raises(ValueError):
        D.threshold(1.0)
    with pytest.raises(ValueError):
        D.threshold(-0.1)


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_fraction(p):
    n = 1024
    z = D.keep_mask(np.arange(n), np.arange(n), 7, p, 99, 3)
    keep = 1.0 - D.threshold(p) / 65536.0
    sigma = np.sqrt(keep * (1 - keep) / z.size)
    assert abs(z.mean() - keep) < 5 * sigma
    # neighbours (same call / same word) are not correlated
    a = z[:, 0::2].astype(np.float64).ravel()
    b = z[:, 1::2].astype(np.float64).ravel()
    assert abs(np.corrcoef(a, b)[0, 1]) < 5 / np.sqrt(a.size)
    # another offset, head or seed gives another mask
    assert np.mean(z != D.keep_mask(np.arange(n), np.arange(n), 7, p, 99, 4)) > 0.05
    assert np.mean(z != D.keep_mask(np.arange(n), np.arange(n), 8, p, 99, 3)) > 0.05
    assert np.mean(z != D.keep_mask(np.arange(n), np.arange(n), 7, p, 98, 3)) > 0.05


def tiny(B=1, H=2, N=40, d=8, seed=0):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, H, N, d)) for _ in range(4)]


def test_zero_probability_is_plain_attention():
    q, k, v, do = tiny()
    o0, l0 = oracle.forward(q, k, v, 0.3, causal=True)
    o1, l1 = oracle.forward(q, k, v, 0.3, causal=True, dropout=(0.0, 5, 1))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    g0 = oracle.backward(q, k, v, do, 0.3, causal=True)
    g1 = oracle.backward(q, k, v, do, 0.3, causal=True, dropout=(0.0, 5, 1))
    for a, b in zip(g0, g1):
        assert np.array_equal(a, b)


def test_expectation_over_seeds_is_plain_attention():
    """E_Z[(P o Z) V / (1-p)] = P V: the mean over many seeds converges to the
    undropped output (standard error shrinking as 1/sqrt(seeds))."""
    q, k, v, _ = tiny(B=1, H=1, N=24, d=4, seed=1)
    o_ref, lse_ref = oracle.forward(q, k, v, 0.5)
    seeds = 3000
    acc = np.zeros_like(o_ref)
    sq = np.zeros_like(o_ref)
    for s in range(seeds):
        o, lse = oracle.forward(q, k, v, 0.5, dropout=(0.4, s, 0))
        assert np.allclose(lse, lse_ref)   # lse is that of the undropped scores
        acc += o
        sq += o * o
    mean = acc / seeds
    se = np.sqrt(np.maximum(sq / seeds - mean * mean, 1e-30) / seeds)
    assert np.all(np.abs(mean - o_ref) < 6 * se + 1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_with_dropout_matches_finite_differences(causal):
    """With the mask fixed by (seed, offset), the loss L = sum(O * dO) is a
    smooth function of Q, K, V; central differences of the oracle's forward
    pin its backward, including where Z and 1/(1-p) enter."""
    B, H, N, d = 1, 1, 12, 4
    q, k, v, do = tiny(B, H, N, d, seed=2)
    drop = (0.3, 1234, 9)
    scale = 0.7
    dq, dk, dv, _ = oracle.backward(q, k, v, do, scale, causal=causal, dropout=drop)

    def loss(q_, k_, v_):
        o, _ = oracle.forward(q_, k_, v_, scale, causal=causal, dropout=drop)
        return float(np.sum(o * do))

    eps = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p, args_m = [q, k, v], [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        assert np.max(np.abs(num - g)) < 1e-6 * max(1.0, np.max(np.abs(g)))


def test_sampled_rows_agree_with_whole_tensor():
    q, k, v, do = tiny(B=2, H=2, N=300, d=8, seed=4)
    drop = (0.2, 77, 5)
    o, lse = oracle.forward(q, k, v, 0.4, causal=True, dropout=drop)
    dq, dk, dv, dd = oracle.backward(q, k, v, do, 0.4, causal=True, dropout=drop)
    rows = np.stack([np.stack([np.array([0, 5, 128, 299])] * 2)] * 2)
    ro, rl = oracle.forward_rows(q, k, v, 0.4, rows, causal=True, dropout=drop)
    assert np.allclose(ro, np.take_along_axis(o, rows[..., None], 2))
    rdq = oracle.backward_query_rows(q, k, v, do, 0.4, rows, causal=True, dropout=drop)
    assert np.allclose(rdq, np.take_along_axis(dq, rows[..., None], 2))
    lse_all, d_all = oracle.row_stats(q, k, v, do, 0.4, causal=True, dropout=drop)
    assert np.allclose(d_all, dd) and np.allclose(lse_all, lse)
    # D_i = dO_i . O_i also holds with dropout
    assert np.allclose(dd, np.sum(do * o, -1))
    rdk, rdv = oracle.backward_key_rows(q, k, v, do, 0.4, rows, lse_all, d_all, causal=True,
                                        dropout=drop)
    assert np.allclose(rdk, np.take_along_axis(dk, rows[..., None], 2))
    assert np.allclose(rdv, np.take_along_axis(dv, rows[..., None], 2))
