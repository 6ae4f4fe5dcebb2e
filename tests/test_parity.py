"""GPU parity: libfa through its C ABI against the fp64 oracle on the same
seeded inputs, element by element, within the stated tolerances
(bf16: O max-abs 1e-2, lse max-abs 1e-3, dQ/dK/dV relative Frobenius 2e-2;
fp32: ten times tighter)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, block_mask_pattern, generate, random_case
from _gpu_helpers import TOL, f64, max_abs, rel_fro, run, to_device
from _oracle_pool import key_rows_every_head

pytestmark = pytest.mark.gpu


def check_full(fa, case, B, H, N, d, causal, dtype, bwd=True):
    scale = d ** -0.5
    t = to_device(case, dtype)
    o, lse, grads = run(fa, t, scale, causal, with_bwd=bwd)
    kw = dict(causal=causal, kv_len=case.get("kv_len"), block_mask=case.get("block_mask"))
    ro, rl = oracle.forward(case["q"], case["k"], case["v"], scale, **kw)
    to, tl, tg = TOL[dtype]
    e_o = max_abs(f64(o), ro)
    e_l = max_abs(lse.cpu().numpy().astype(np.float64), rl, finite_only=True)
    assert np.array_equal(np.isneginf(lse.cpu().numpy()), np.isneginf(rl)), "empty-row pattern"
    assert e_o <= to, ("O", e_o)
    assert e_l <= tl, ("lse", e_l)
    if bwd:
        rdq, rdk, rdv, _ = oracle.backward(case["q"], case["k"], case["v"], case["do"], scale, **kw)
        for name, g, r in zip(("dQ", "dK", "dV"), grads, (rdq, rdk, rdv)):
            e = rel_fro(f64(g), r)
            assert e <= tg, (name, e)
    return o, lse, grads


SMALL = [
    # B, H, N, d, causal, mask
    (1, 2, 128, 64, False, "none"),
    (1, 2, 128, 128, True, "none"),
    (2, 2, 300, 64, True, "none"),        # ragged tail
    (1, 1, 1, 64, False, "none"),         # a single token
    (1, 2, 77, 128, False, "none"),       # shorter than one tile
    (1, 1, 1000, 64, True, "none"),       # many tiles, ragged
    (1, 2, 513, 128, False, "none"),
    (2, 3, 384, 64, False, "padding"),
    (2, 2, 512, 128, True, "padding"),
    (1, 2, 640, 64, False, "sparse"),
    (1, 2, 520, 128, True, "sparse"),
    # d = 64 kernels walk 64-row / 64-key half steps: tails inside either half,
    # causal with each mask kind
    (2, 2, 200, 64, False, "none"),       # second half of the last tile partly past N
    (1, 2, 1000, 64, False, "padding"),
    (2, 2, 333, 64, True, "padding"),
    (1, 2, 520, 64, True, "sparse"),
]


def small_case(B, H, N, d, mask, seed, dtype="bf16"):
    rng = np.random.default_rng(seed + 99)
    kv = bm = None
    if mask == "padding":
        kv = rng.integers(1, N + 1, B)
        kv[0] = min(N, 100)
    if mask == "sparse":
        T = (N + 127) // 128
        bm = (rng.random((T, T)) < 0.35).astype(np.uint8)
        bm[np.arange(T), np.arange(T)] = 1
    return random_case(B, H, N, d, seed, dtype=dtype, kv_len=kv, block_mask=bm)


@pytest.mark.parametrize("B,H,N,d,causal,mask", SMALL)
def test_small_bf16(fa, B, H, N, d, causal, mask):
    case = small_case(B, H, N, d, mask, seed=N + d)
    check_full(fa, case, B, H, N, d, causal, "bf16")


@pytest.mark.parametrize("B,H,N,d,causal,mask", [
    (1, 2, 256, 64, False, "none"), (1, 2, 256, 64, True, "none"),
    (1, 2, 200, 128, True, "none"), (2, 2, 300, 64, False, "padding"),
    (1, 2, 384, 64, False, "sparse"),
])
def test_small_fp32(fa, B, H, N, d, causal, mask):
    case = small_case(B, H, N, d, mask, seed=N + d + 1, dtype="fp32")
    check_full(fa, case, B, H, N, d, causal, "fp32")


def test_max_heads(fa):
    """B*H = 65535, the largest the library takes: every kernel's grid at its
    widest (the last group of heads in the grid order is ragged), every
    (batch, head) against the oracle.  N = 3, causal: row 0 sees one key.
    With so few keys a row of O is close to one row of V, and over 12.6M
    unit-normal values |O| reaches 4, where bf16's half ulp (2^-6) alone is
    above the absolute O tolerance; values at a quarter keep |O| < 2."""
    B, H, N, d = 257, 255, 3, 64
    case = random_case(B, H, N, d, seed=65535, value_scale=0.25)
    check_full(fa, case, B, H, N, d, True, "bf16")


def test_empty_rows(fa):
    """Block-sparse rows with no visible tile: O = 0, lse = -inf, no gradient."""
    B, H, N, d = 1, 2, 384, 64
    bm = np.array([[0, 0, 0], [1, 1, 0], [0, 1, 1]], np.uint8)
    case = random_case(B, H, N, d, seed=3, block_mask=bm)
    o, lse, grads = check_full(fa, case, B, H, N, d, False, "bf16")
    assert torch.all(o[:, :, :128] == 0)
    assert torch.all(torch.isneginf(lse[:, :, :128]))


@pytest.mark.parametrize("d", [64, 128])
def test_unseen_key_tiles_and_all_padding(fa, d):
    """Key tiles that no query tile sees (an all-zero block-mask column: a dK/dV
    CTA with no work, dK = dV = 0), and a batch whose keys are all padding
    (kv_len = 0: O = 0, lse = -inf, no gradient anywhere in that batch)."""
    B, H, N = 2, 2, 512
    bm = np.array([[1, 0, 0, 1], [1, 0, 1, 0], [0, 0, 1, 1], [1, 0, 0, 1]], np.uint8)
    case = random_case(1, H, N, d, seed=41 + d, block_mask=bm)
    o, lse, (dq, dk, dv) = check_full(fa, case, 1, H, N, d, False, "bf16")
    assert torch.all(dk[:, :, 128:256] == 0) and torch.all(dv[:, :, 128:256] == 0)
    case = random_case(B, H, N, d, seed=43 + d, kv_len=np.array([0, 300], np.int32))
    for causal in (False, True):
        o, lse, (dq, dk, dv) = check_full(fa, case, B, H, N, d, causal, "bf16")
        assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
        assert torch.all(dq[0] == 0) and torch.all(dk[0] == 0) and torch.all(dv[0] == 0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_lengths_at_step_boundaries(fa, d, causal):
    """Key lengths at and beside the 64-key step and 128-key tile boundaries:
    the d = 64 dQ CTA skips a step whose 64 keys all lie past the length (64,
    192: the last tile's second half empty; 65, 129: one key in it), and the
    dK/dV CTAs of tiles past the length write zero rows and leave before
    set-up (1: three of the four tiles; 128, 256: whole tiles)."""
    N = 512
    kv = np.array([64, 65, 127, 128, 129, 192, 1, 256], np.int32)
    case = random_case(len(kv), 2, N, d, seed=61 + d + causal, kv_len=kv)
    o, lse, (dq, dk, dv) = check_full(fa, case, len(kv), 2, N, d, causal, "bf16")
    for bi, L in enumerate(kv):
        assert torch.all(dk[bi, :, L:] == 0) and torch.all(dv[bi, :, L:] == 0)


@pytest.mark.parametrize("name", ["tiny_fp32", "tiny_fp32_causal"])
def test_workload_tiny_fp32(fa, name):
    w = WORKLOADS[name]
    case = generate(w)
    check_full(fa, case, w.B, w.H, w.N, w.d, w.causal, "fp32")


@pytest.mark.parametrize("name", ["gpt2_causal", "bert_padding"])
def test_workload_full(fa, name):
    w = WORKLOADS[name]
    case = generate(w)
    check_full(fa, case, w.B, w.H, w.N, w.d, w.causal, "bf16")


def test_forward_is_deterministic(fa):
    case = random_case(1, 2, 1000, 128, seed=11)
    t = to_device(case, "bf16")
    o1, l1 = fa.forward(t["q"], t["k"], t["v"], 128 ** -0.5, True)
    o2, l2 = fa.forward(t["q"], t["k"], t["v"], 128 ** -0.5, True)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_backward_is_deterministic(fa):
    # every dQ, dK, dV row is summed by one CTA in a fixed order: no atomics
    case = random_case(2, 3, 1000, 128, seed=12)
    t = to_device(case, "bf16")
    scale = 128 ** -0.5
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, True)
    g1 = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, True)
    g2 = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, True)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------------------
# long workloads: sampled rows -- O, lse, dQ on 256 query rows of every head;
# dK, dV on 256 key rows of every head, which need the oracle's statistics of
# every query row of the head (computed a head per host core) -- plus
# properties that hold at any size
# ---------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("name", ["long_causal_d128", "block_sparse", "sparse_local_global",
                                  "sparse_butterfly"])
def test_workload_sampled(fa, name):
    w = WORKLOADS[name]
    case = generate(w)
    scale = w.scale
    t = to_device(case, "bf16")
    o, lse, (dq, dk, dv) = run(fa, t, scale, w.causal)
    kw = dict(causal=w.causal, kv_len=case["kv_len"], block_mask=case["block_mask"])
    rows, cols = case["rows"], case["cols"]
    to, tl, tg = TOL["bf16"]
    take = lambda a, r: np.take_along_axis(a, r[..., None], axis=2)
    ro, rl = oracle.forward_rows(case["q"], case["k"], case["v"], scale, rows, **kw)
    assert max_abs(take(f64(o), rows), ro) <= to
    assert max_abs(np.take_along_axis(lse.cpu().numpy().astype(np.float64), rows, axis=2), rl) <= tl
    rdq = oracle.backward_query_rows(case["q"], case["k"], case["v"], case["do"], scale, rows, **kw)
    assert rel_fro(take(f64(dq), rows), rdq) <= tg
    lse_all, rdk, rdv = key_rows_every_head(case["q"], case["k"], case["v"], case["do"], scale,
                                            cols, **kw)
    assert rel_fro(take(f64(dk), cols), rdk) <= tg
    assert rel_fro(take(f64(dv), cols), rdv) <= tg
    # per head too, so that one wrong head cannot hide among the others
    for b in range(w.B):
        for h in range(w.H):
            assert rel_fro(take(f64(dk), cols)[b, h], rdk[b, h]) <= tg, ("dK", b, h)
            assert rel_fro(take(f64(dv), cols)[b, h], rdv[b, h]) <= tg, ("dV", b, h)
    # the oracle's lse of every row against the GPU's
    assert max_abs(lse.cpu().numpy().astype(np.float64), lse_all) <= tl
    # any size: shifting every key by one vector leaves O unchanged, so the
    # key gradients of each head sum to zero (bf16 rounding allows a little)
    dk64 = f64(dk)
    tot = np.linalg.norm(dk64.sum(axis=2), axis=-1)
    per = np.linalg.norm(dk64, axis=(2, 3))
    assert np.all(tot <= 2e-2 * per)
    # any size: every row sees a key and its probabilities sum to one, so the
    # value gradients of each head sum to its dO summed over the rows
    dv64 = f64(dv)
    err = np.linalg.norm(dv64.sum(axis=2) - case["do"].sum(axis=2), axis=-1)
    assert np.all(err <= 2e-2 * np.linalg.norm(dv64, axis=(2, 3)))


@pytest.mark.parametrize("pattern", ["local", "local_global", "strided", "butterfly"])
@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_sparse_patterns(fa, pattern, d, causal):
    """Every structured tile pattern, all rows against the oracle (T = 16)."""
    B, H, N = 1, 2, 2048 - 37   # ragged last tile
    T = (N + 127) // 128
    case = random_case(B, H, N, d, seed=sum(map(ord, pattern)) + d,
                       block_mask=block_mask_pattern(pattern, T))
    check_full(fa, case, B, H, N, d, causal, "bf16")


@pytest.mark.slow
def test_path256_butterfly(fa):
    """Path-256 length (65536 tokens) under the butterfly tile mask: sampled
    query rows, and every row of one key tile exactly (the oracle needs the
    statistics of just the query tiles that see it)."""
    B, H, N, d = 1, 2, 65536, 64
    T = N // 128
    bm = block_mask_pattern("butterfly", T)
    case = random_case(B, H, N, d, seed=256, block_mask=bm)
    scale = d ** -0.5
    t = to_device(case, "bf16")
    o, lse, (dq, dk, dv) = run(fa, t, scale, False)
    to, tl, tg = TOL["bf16"]
    kw = dict(block_mask=bm)
    rng = np.random.default_rng(256)
    rows = np.stack([np.stack([np.sort(rng.choice(N, 256, replace=False)) for _ in range(H)])
                     for _ in range(B)])
    take = lambda a, r: np.take_along_axis(a, r[..., None], axis=2)
    ro, rl = oracle.forward_rows(case["q"], case["k"], case["v"], scale, rows, **kw)
    assert max_abs(take(f64(o), rows), ro) <= to
    assert max_abs(np.take_along_axis(lse.cpu().numpy().astype(np.float64), rows, axis=2),
                   rl) <= tl
    rdq = oracle.backward_query_rows(case["q"], case["k"], case["v"], case["do"], scale, rows,
                                     **kw)
    assert rel_fro(take(f64(dq), rows), rdq) <= tg
    kt = 300
    seen_by = np.flatnonzero(bm[:, kt])
    qrows = np.concatenate([np.arange(i * 128, i * 128 + 128) for i in seen_by])
    qrows = np.broadcast_to(qrows, (B, H, qrows.size)).copy()
    so, sl = oracle.forward_rows(case["q"], case["k"], case["v"], scale, qrows, **kw)
    lse_all = np.zeros((B, H, N))
    d_all = np.zeros((B, H, N))
    np.put_along_axis(lse_all, qrows, sl, axis=2)
    do_rows = np.take_along_axis(np.asarray(case["do"], np.float64), qrows[..., None], axis=2)
    np.put_along_axis(d_all, qrows, np.sum(do_rows * so, -1), axis=2)
    keys = np.broadcast_to(np.arange(kt * 128, kt * 128 + 128), (B, H, 128)).copy()
    rdk, rdv = oracle.backward_key_rows(case["q"], case["k"], case["v"], case["do"], scale, keys,
                                        lse_all, d_all, **kw)
    assert rel_fro(f64(dk)[..., kt * 128:kt * 128 + 128, :], rdk) <= tg
    assert rel_fro(f64(dv)[..., kt * 128:kt * 128 + 128, :], rdv) <= tg
    dk64 = f64(dk)
    tot = np.linalg.norm(dk64.sum(axis=2), axis=-1)
    per = np.linalg.norm(dk64, axis=(2, 3))
    assert np.all(tot <= 2e-2 * per)


# ---------------------------------------------------------------------------
# 64K-token causal contexts.  Query rows: 256 sampled per head (O, lse, dQ).
# Key rows: the last key tile, exactly -- under the causal mask only the last
# 128 query rows see those keys, so the oracle needs the statistics (lse, D)
# of those rows only.
# ---------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("d", [128, 64])
def test_causal_64k(fa, d):
    B, H, N = 1, 2, 65536
    case = random_case(B, H, N, d, seed=21 + d, value_scale=0.5)
    scale = d ** -0.5
    t = to_device(case, "bf16")
    o, lse, (dq, dk, dv) = run(fa, t, scale, True)
    to, tl, tg = TOL["bf16"]
    rng = np.random.default_rng(64)
    rows = np.stack([np.stack([np.sort(np.concatenate(
        [[0, 127, 128, N - 1], rng.choice(np.arange(129, N - 1), 252, replace=False)]))
        for _ in range(H)]) for _ in range(B)])
    take = lambda a, r: np.take_along_axis(a, r[..., None], axis=2)
    ro, rl = oracle.forward_rows(case["q"], case["k"], case["v"], scale, rows, causal=True)
    assert max_abs(take(f64(o), rows), ro) <= to
    assert max_abs(np.take_along_axis(lse.cpu().numpy().astype(np.float64), rows, axis=2),
                   rl) <= tl
    rdq = oracle.backward_query_rows(case["q"], case["k"], case["v"], case["do"], scale, rows,
                                     causal=True)
    assert rel_fro(take(f64(dq), rows), rdq) <= tg
    last = np.broadcast_to(np.arange(N - 128, N), (B, H, 128)).copy()
    lo, ll = oracle.forward_rows(case["q"], case["k"], case["v"], scale, last, causal=True)
    lse_all = np.zeros((B, H, N))
    d_all = np.zeros((B, H, N))
    lse_all[..., N - 128:] = ll
    d_all[..., N - 128:] = np.sum(np.asarray(case["do"][..., N - 128:, :], np.float64) * lo, -1)
    rdk, rdv = oracle.backward_key_rows(case["q"], case["k"], case["v"], case["do"], scale, last,
                                        lse_all, d_all, causal=True)
    assert rel_fro(f64(dk)[..., N - 128:, :], rdk) <= tg
    assert rel_fro(f64(dv)[..., N - 128:, :], rdv) <= tg
    # any size: the key gradients of each head sum to zero
    dk64 = f64(dk)
    tot = np.linalg.norm(dk64.sum(axis=2), axis=-1)
    per = np.linalg.norm(dk64, axis=(2, 3))
    assert np.all(tot <= 2e-2 * per)
