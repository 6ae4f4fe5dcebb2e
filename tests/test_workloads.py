"""CPU checks of the seeded input generators: shapes, determinism, and the
structure of each block-sparse tile pattern."""
import numpy as np
import pytest

from workloads import PATTERNS, WORKLOADS, block_mask_pattern, generate


@pytest.mark.parametrize("pattern", PATTERNS)
@pytest.mark.parametrize("T", [1, 5, 64, 128])
def test_patterns_keep_the_diagonal(pattern, T):
    m = block_mask_pattern(pattern, T, np.random.default_rng(0))
    assert m.shape == (T, T) and m.dtype == np.uint8
    assert set(np.unique(m)) <= {0, 1}
    assert np.all(np.diag(m) == 1)


def test_band_patterns():
    T = 40
    i, j = np.indices((T, T))
    assert np.array_equal(block_mask_pattern("local", T), (abs(i - j) <= 2).astype(np.uint8))
    lg = block_mask_pattern("local_global", T)
    assert lg[0].all() and lg[:, 0].all()
    assert np.array_equal(lg[1:, 1:], (abs(i - j) <= 1)[1:, 1:].astype(np.uint8))
    st = block_mask_pattern("strided", T)
    assert st[:, 7::8].all()
    assert st.sum() == ((abs(i - j) <= 1) | (j % 8 == 7)).sum()


@pytest.mark.parametrize("T", [8, 128, 512])
def test_butterfly_pattern(T):
    m = block_mask_pattern("butterfly", T)
    # symmetric, 1 + log2(T) tiles per row: the diagonal and one partner per bit
    assert np.array_equal(m, m.T)
    assert np.all(m.sum(axis=1) == 1 + int(np.log2(T)))
    for i in (0, 3, T - 1):
        partners = sorted(int(j) for j in np.flatnonzero(m[i]) if j != i)
        assert partners == sorted(i ^ (1 << b) for b in range(int(np.log2(T))))


def test_random_pattern_is_the_seeded_draw():
    a = generate("block_sparse")["block_mask"]
    b = generate("block_sparse")["block_mask"]
    assert np.array_equal(a, b)
    assert 0.10 < a.mean() < 0.16   # p = 0.125 plus the diagonal


@pytest.mark.parametrize("name", ["sparse_local_global", "sparse_butterfly"])
def test_structured_workloads(name):
    w = WORKLOADS[name]
    g = generate(w, samples=4)
    assert g["block_mask"].shape == (w.tiles, w.tiles)
    assert np.array_equal(g["block_mask"], block_mask_pattern(w.pattern, w.tiles))
    assert g["q"].shape == (w.B, w.H, w.N, w.d)
