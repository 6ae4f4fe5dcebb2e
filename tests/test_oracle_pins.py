"""Pins for the fp64 oracle: each checks it against something other than
itself -- closed forms, invariants the pages derive, hand-derived values,
brute force, finite differences and an independent autograd.

Sources (page title, section):
  * "From Online Softmax to FlashAttention" (blog review): "(safe) softmax"
    (3-pass algorithm), "Online Softmax" (2-pass), "Algorithm FlashAttention
    (Tiling)", and the d = 1 specification function at "The Self-Attention".
  * "FlashAttention: Fast and Memory-Efficient Exact Attention with
    IO-Awareness" (summary page): "Problem and motivation" (definition),
    "Extension: block-sparse FlashAttention".
  * GitHub issue "Fewer matrix multiplications, same results": causal
    lower-triangular mask and the 1/sqrt(d) scale on the scores.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import attention as A

HERE = os.path.dirname(os.path.abspath(__file__))


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


MASKS = ["none", "causal", "padding", "sparse", "causal_sparse", "causal_padding"]


def mask_args(kind, B, N, seed, block):
    rng = np.random.default_rng(seed + 1000)
    causal = kind.startswith("causal")
    kv_len = None
    bm = None
    if "padding" in kind:
        kv_len = rng.integers(1, N + 1, B)
    if "sparse" in kind:
        T = (N + block - 1) // block
        bm = (rng.random((T, T)) < 0.5).astype(np.uint8)
        bm[np.arange(T), np.arange(T)] = 1
    return dict(causal=causal, kv_len=kv_len, block_mask=bm, block=block)


# ---------------------------------------------------------------------------
# 1. softmax rows sum to 1
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", MASKS)
def test_probability_rows_sum_to_one(kind):
    N, d = 37, 8
    q, k = rand((N, d), 1), rand((N, d), 2)
    ma = mask_args(kind, 1, N, 3, block=8)
    vis = A.visible(N, N, ma["causal"], None if ma["kv_len"] is None else ma["kv_len"][0],
                    ma["block_mask"], ma["block"])
    p, lse = A.probabilities(A.scores(q, k, 0.35, vis))
    has = vis.any(axis=1)
    assert np.all(np.abs(p.sum(axis=1)[has] - 1.0) <= 1e-12)
    assert np.all(p[~vis] == 0.0)
    assert np.all(p >= 0.0)


def test_empty_row_reading():
    """A row with no visible key: P = 0, O = 0, lse = -inf, no gradient."""
    N, d = 8, 4
    q, k, v, do = (rand((1, 1, N, d), s) for s in range(4))
    bm = np.zeros((2, 2), np.uint8)
    bm[1, 1] = 1   # query rows 0..3 see nothing
    o, lse = A.forward(q, k, v, 0.5, block_mask=bm, block=4)
    assert np.all(o[0, 0, :4] == 0.0) and np.all(np.isneginf(lse[0, 0, :4]))
    dq, dk, dv, _ = A.backward(q, k, v, do, 0.5, block_mask=bm, block=4)
    assert np.all(dq[0, 0, :4] == 0.0)
    assert np.all(dk[0, 0, :4] == 0.0) and np.all(dv[0, 0, :4] == 0.0)


# ---------------------------------------------------------------------------
# 2. 3-pass safe softmax == 2-pass online softmax == tiled 1-pass recurrence
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("offset", [0.0, 1e4, -1e4, 37.5])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_three_pass_equals_online(offset, seed):
    x = rand(50, seed, 4.0) + offset
    a3, m3, d3 = A.softmax_three_pass(x)
    a2, m2, d2 = A.softmax_online_two_pass(x)
    assert m3 == m2 == np.max(x)
    assert abs(d3 - d2) <= 1e-12 * d3
    assert np.max(np.abs(a3 - a2)) <= 1e-12
    assert abs(a3.sum() - 1.0) <= 1e-12
    # and both equal the oracle's softmax of the row
    p, lse = A.probabilities(x[None, :])
    assert np.max(np.abs(p[0] - a3)) <= 1e-12
    assert abs(lse[0] - (m3 + math.log(d3))) <= 1e-9 * max(1.0, abs(lse[0]))


@pytest.mark.parametrize("seed", range(6))
def test_tiled_one_pass_equals_definition(seed):
    rng = np.random.default_rng(seed)
    N, d = 97, 5
    x = rng.standard_normal(N) * 3.0 + rng.uniform(-50, 50)
    v = rng.standard_normal((N, d))
    cuts = sorted(set(rng.choice(np.arange(1, N), size=rng.integers(0, 12), replace=False)))
    starts = [0] + list(cuts)
    o, m, dsum = A.attention_row_one_pass_tiled(x, v, starts)
    p, lse = A.probabilities(x[None, :])
    assert np.max(np.abs(o - p[0] @ v)) <= 1e-12
    assert m == np.max(x)
    assert abs(m + math.log(dsum) - lse[0]) <= 1e-12 * max(1.0, abs(lse[0]))


# ---------------------------------------------------------------------------
# 3. causal: row 0 sees key 0 only
# ---------------------------------------------------------------------------

def test_causal_row_zero():
    B, H, N, d = 2, 3, 40, 16
    q, k, v = rand((B, H, N, d), 1), rand((B, H, N, d), 2), rand((B, H, N, d), 3)
    s = 0.25
    o, lse = A.forward(q, k, v, s, causal=True)
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0])) <= 1e-15
    expect = s * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    assert np.max(np.abs(lse[:, :, 0] - expect)) <= 1e-13


# ---------------------------------------------------------------------------
# 4. identical keys: uniform attention over the visible keys
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", MASKS)
def test_identical_keys_mean_of_visible_values(kind):
    B, H, N, d = 2, 2, 24, 6
    q, v = rand((B, H, N, d), 5), rand((B, H, N, d), 6)
    k = np.broadcast_to(rand((B, H, 1, d), 7), (B, H, N, d)).copy()
    s = 0.7
    ma = mask_args(kind, B, N, 8, block=8)
    o, lse = A.forward(q, k, v, s, **ma)
    for b in range(B):
        kv = None if ma["kv_len"] is None else ma["kv_len"][b]
        vis = A.visible(N, N, ma["causal"], kv, ma["block_mask"], 8)
        for h in range(H):
            for i in range(N):
                cnt = vis[i].sum()
                if cnt == 0:
                    assert np.all(o[b, h, i] == 0) and np.isneginf(lse[b, h, i])
                    continue
                mean = v[b, h][vis[i]].mean(axis=0)
                assert np.max(np.abs(o[b, h, i] - mean)) <= 1e-13
                want = s * q[b, h, i] @ k[b, h, 0] + math.log(cnt)
                assert abs(lse[b, h, i] - want) <= 1e-12


# ---------------------------------------------------------------------------
# 5. all-ones block mask == dense; padding with L = N == dense
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_trivial_masks_equal_dense(causal):
    B, H, N, d = 2, 2, 50, 8
    q, k, v, do = (rand((B, H, N, d), s) for s in range(10, 14))
    o0, l0 = A.forward(q, k, v, 0.3, causal=causal)
    g0 = A.backward(q, k, v, do, 0.3, causal=causal)
    T = (N + 15) // 16
    o1, l1 = A.forward(q, k, v, 0.3, causal=causal, block_mask=np.ones((T, T), np.uint8), block=16)
    o2, l2 = A.forward(q, k, v, 0.3, causal=causal, kv_len=np.full(B, N))
    g1 = A.backward(q, k, v, do, 0.3, causal=causal, block_mask=np.ones((T, T), np.uint8), block=16)
    for a, b_ in [(o0, o1), (o0, o2), (l0, l1), (l0, l2)] + list(zip(g0, g1)):
        assert np.array_equal(a, b_)


# ---------------------------------------------------------------------------
# 6. finite differences of L = sum(O * dO)
# ---------------------------------------------------------------------------

def _fd_check(backward_fn, kind, seed, N=12, d=6, h=1e-6):
    B, H = 1, 2
    q, k, v, do = (rand((B, H, N, d), seed + i) for i in range(4))
    s = 1.0 / math.sqrt(d)
    ma = mask_args(kind, B, N, seed, block=4)
    dq, dk, dv, _ = backward_fn(q, k, v, do, s, **ma)

    def loss(q_, k_, v_):
        o, _ = A.forward(q_, k_, v_, s, **ma)
        return float(np.sum(o * do))

    worst = 0.0
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                        loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(num), 1e-30)
        worst = max(worst, err)
    return worst


@pytest.mark.parametrize("kind", MASKS)
def test_gradients_match_finite_differences(kind):
    assert _fd_check(A.backward, kind, seed=21) <= 1e-6


def _mutant(which):
    """A copy of the backward with one plausible mistake planted in it."""
    def bwd(q, k, v, do, scale, causal=False, kv_len=None, block_mask=None, block=128):
        B, H, N, d = q.shape
        out = [np.zeros((B, H, N, d)) for _ in range(3)]
        for b in range(B):
            vis = A.visible(N, N, causal, None if kv_len is None else kv_len[b], block_mask, block)
            for hh in range(H):
                qq, kk, vv, dd = q[b, hh], k[b, hh], v[b, hh], do[b, hh]
                p, _ = A.probabilities(A.scores(qq, kk, scale, vis))
                dv = (p @ dd) if which == "dv_untransposed" else p.T @ dd
                dp = dd @ vv.T
                drow = np.sum(p * dp, axis=1)
                ds = p * dp if which == "drop_D" else p * (dp - drow[:, None])
                sc = 1.0 if which == "dq_no_scale" else scale
                dq = sc * (ds @ kk)
                dk = scale * ((ds @ qq) if which == "dk_untransposed" else ds.T @ qq)
                if which == "dk_sign":
                    dk = -dk
                out[0][b, hh], out[1][b, hh], out[2][b, hh] = dq, dk, dv
        return out[0], out[1], out[2], None
    return bwd


@pytest.mark.parametrize("which", ["dv_untransposed", "drop_D", "dq_no_scale",
                                   "dk_untransposed", "dk_sign"])
def test_finite_differences_catch_planted_mistakes(which):
    """The finite-difference pin is strong enough to reject each of these."""
    assert _fd_check(_mutant(which), "causal", seed=5) > 1e-3


# ---------------------------------------------------------------------------
# 7. d = 1, scale = 1: the blog review's specification function
# ---------------------------------------------------------------------------

def _spec_d1(q, k, v):
    # the blog's specification written independently: outer product of the
    # query and key vectors, row max removed, exponentiated, normalised, and
    # used to average v
    x = np.outer(q, k)
    x = x - x.max(axis=1, keepdims=True)
    w = np.exp(x)
    w = w / w.sum(axis=1, keepdims=True)
    return (w * v[None, :]).sum(axis=1)


def test_d1_matches_specification_function():
    n = 200
    q, k, v = rand(n, 31), rand(n, 32), rand(n, 33)
    o, _ = A.forward(q.reshape(1, 1, n, 1), k.reshape(1, 1, n, 1), v.reshape(1, 1, n, 1), 1.0)
    assert np.max(np.abs(o[0, 0, :, 0] - _spec_d1(q, k, v))) <= 1e-13


# ---------------------------------------------------------------------------
# 8. shift invariance: k_j -> k_j + u adds s q_i.u to every logit of row i
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", MASKS)
def test_shift_invariance(kind):
    B, H, N, d = 2, 2, 30, 8
    q, k, v = rand((B, H, N, d), 40), rand((B, H, N, d), 41), rand((B, H, N, d), 42)
    u = rand((B, H, 1, d), 43, 3.0)
    s = 0.4
    ma = mask_args(kind, B, N, 44, block=8)
    o0, l0 = A.forward(q, k, v, s, **ma)
    o1, l1 = A.forward(q, k + u, v, s, **ma)
    shift = s * np.einsum("bhnd,bhd->bhn", q, u[:, :, 0])
    fin = np.isfinite(l0)
    assert np.max(np.abs(o1 - o0)) <= 1e-12
    assert np.max(np.abs((l1 - l0 - shift)[fin])) <= 1e-11


# ---------------------------------------------------------------------------
# 9. padded keys get exactly zero gradient; 10. sum of dK over keys is zero
# ---------------------------------------------------------------------------

def test_padded_keys_have_zero_gradient():
    B, H, N, d = 3, 2, 33, 8
    q, k, v, do = (rand((B, H, N, d), 50 + i) for i in range(4))
    kv_len = np.array([5, 33, 17])
    _, dk, dv, _ = A.backward(q, k, v, do, 0.3, kv_len=kv_len)
    for b in range(B):
        assert np.all(dk[b, :, kv_len[b]:] == 0.0)
        assert np.all(dv[b, :, kv_len[b]:] == 0.0)


@pytest.mark.parametrize("kind", MASKS)
def test_dk_sums_to_zero(kind):
    B, H, N, d = 2, 2, 40, 8
    q, k, v, do = (rand((B, H, N, d), 60 + i) for i in range(4))
    ma = mask_args(kind, B, N, 64, block=8)
    _, dk, _, _ = A.backward(q, k, v, do, 0.3, **ma)
    tot = dk.sum(axis=2)
    assert np.max(np.abs(tot)) <= 1e-10 * max(1.0, np.linalg.norm(dk))


@pytest.mark.parametrize("kind", MASKS)
def test_dv_sums_to_the_summed_do(kind):
    """Every row of P sums to one and dV = P^T dO, so the value gradients of a
    head sum to its dO summed over the rows (every row here sees a key).  A
    transposed P in dV, or a dropped row, breaks it."""
    B, H, N, d = 2, 2, 40, 8
    q, k, v, do = (rand((B, H, N, d), 70 + i) for i in range(4))
    ma = mask_args(kind, B, N, 65, block=8)
    _, _, dv, _ = A.backward(q, k, v, do, 0.3, **ma)
    err = np.max(np.abs(dv.sum(axis=2) - do.sum(axis=2)))
    assert err <= 1e-10 * max(1.0, np.linalg.norm(dv))


# ---------------------------------------------------------------------------
# 11. hand-derived values
# ---------------------------------------------------------------------------

def _num(x):
    if isinstance(x, (int, float)):
        return float(x)
    table = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4),
             "ln5": math.log(5), "ln6": math.log(6), "-ln2/4": -math.log(2) / 4,
             "ln3/8": math.log(3) / 8}
    if x in table:
        return table[x]
    return float(Fraction(x))


def _arr(a):
    return np.array([[_num(e) for e in row] if isinstance(row, list) else _num(row) for row in a])


def test_hand_derived_golden_values():
    g = json.load(open(os.path.join(HERE, "golden", "hand_n3_d2.json")))
    q, k, v = (_arr(g[n]).reshape(1, 1, 3, 2) for n in ("q", "k", "v"))
    s = g["scale"]
    o, lse = A.forward(q, k, v, s)
    assert np.max(np.abs(o[0, 0] - _arr(g["noncausal"]["o"]))) <= 1e-15
    assert np.max(np.abs(lse[0, 0] - _arr(g["noncausal"]["lse"]))) <= 1e-15
    o, lse = A.forward(q, k, v, s, causal=True)
    assert np.max(np.abs(o[0, 0] - _arr(g["causal"]["o"]))) <= 1e-15
    assert np.max(np.abs(lse[0, 0] - _arr(g["causal"]["lse"]))) <= 1e-15
    do = _arr(g["backward_noncausal"]["do"]).reshape(1, 1, 3, 2)
    dq, dk, dv, _ = A.backward(q, k, v, do, s)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert np.max(np.abs(got[0, 0] - _arr(g["backward_noncausal"][name]))) <= 1e-15, name


# ---------------------------------------------------------------------------
# 12. brute force with scalar loops on tiny inputs
# ---------------------------------------------------------------------------

def _brute(q, k, v, s, vis):
    n, d = len(q), len(q[0])
    o = [[0.0] * d for _ in range(n)]
    lse = [0.0] * n
    for i in range(n):
        logits = [s * sum(q[i][c] * k[j][c] for c in range(d)) for j in range(n) if vis[i][j]]
        idx = [j for j in range(n) if vis[i][j]]
        mx = max(logits)
        w = [math.exp(x - mx) for x in logits]
        tot = sum(w)
        lse[i] = mx + math.log(tot)
        for c in range(d):
            o[i][c] = sum(w[t] / tot * v[idx[t]][c] for t in range(len(idx)))
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("kind", ["none", "causal", "padding", "sparse"])
def test_brute_force_loops(kind):
    N, d = 9, 3
    q, k, v = rand((1, 1, N, d), 70), rand((1, 1, N, d), 71), rand((1, 1, N, d), 72)
    ma = mask_args(kind, 1, N, 73, block=4)
    if ma["kv_len"] is not None:
        ma["kv_len"] = np.array([6])
    o, lse = A.forward(q, k, v, 0.6, **ma)
    vis = A.visible(N, N, ma["causal"], None if ma["kv_len"] is None else 6, ma["block_mask"], 4)
    ob, lb = _brute(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), 0.6, vis.tolist())
    assert np.max(np.abs(o[0, 0] - ob)) <= 1e-13
    assert np.max(np.abs(lse[0, 0] - lb)) <= 1e-13


# ---------------------------------------------------------------------------
# 13. independent autograd (torch CPU, float64) of the naive formula
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", MASKS)
def test_torch_autograd_cross_check(kind):
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 2, 48, 16
    q, k, v, do = (rand((B, H, N, d), 80 + i) for i in range(4))
    s = 0.25
    ma = mask_args(kind, B, N, 85, block=16)
    o, lse = A.forward(q, k, v, s, **ma)
    dq, dk, dv, _ = A.backward(q, k, v, do, s, **ma)
    vis = np.stack([A.visible(N, N, ma["causal"], None if ma["kv_len"] is None else ma["kv_len"][b],
                              ma["block_mask"], 16) for b in range(B)])
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    logits = s * tq @ tk.transpose(-1, -2)
    logits = logits.masked_fill(~torch.tensor(vis)[:, None], float("-inf"))
    has = torch.tensor(vis.any(axis=2))[:, None, :, None]
    p = torch.softmax(logits, dim=-1).nan_to_num(0.0) * has
    to = p @ tv
    (to * torch.tensor(do)).sum().backward()
    assert np.max(np.abs(to.detach().numpy() - o)) <= 1e-12
    tl = torch.logsumexp(logits, dim=-1).detach().numpy()
    assert np.allclose(tl, lse, atol=1e-12, rtol=0)
    for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.max(np.abs(got - ref.numpy())) <= 1e-11


# ---------------------------------------------------------------------------
# 14. sampled-row paths agree with the full computation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["causal", "sparse", "padding"])
def test_sampled_rows_equal_full(kind):
    B, H, N, d = 2, 2, 70, 8
    q, k, v, do = (rand((B, H, N, d), 90 + i) for i in range(4))
    s = 0.3
    ma = mask_args(kind, B, N, 95, block=16)
    o, lse = A.forward(q, k, v, s, **ma)
    dq, dk, dv, dd = A.backward(q, k, v, do, s, **ma)
    rng = np.random.default_rng(3)
    rows = np.stack([np.stack([rng.choice(N, 11, replace=False) for _ in range(H)]) for _ in range(B)])
    cols = np.stack([np.stack([rng.choice(N, 13, replace=False) for _ in range(H)]) for _ in range(B)])
    take = lambda a, r: np.take_along_axis(a, r[..., None] if a.ndim == 4 else r, axis=2)
    o_r, lse_r = A.forward_rows(q, k, v, s, rows, **ma)
    assert np.max(np.abs(o_r - take(o, rows))) <= 1e-13
    fin = np.isfinite(take(lse, rows))
    assert np.max(np.abs((lse_r - take(lse, rows))[fin])) <= 1e-13
    dq_r = A.backward_query_rows(q, k, v, do, s, rows, **ma)
    assert np.max(np.abs(dq_r - take(dq, rows))) <= 1e-12
    lse_all, dd_all = A.row_stats(q, k, v, do, s, rows_per_group=16, **ma)
    assert np.max(np.abs(dd_all - dd)) <= 1e-12
    dk_c, dv_c = A.backward_key_rows(q, k, v, do, s, cols, lse_all, dd_all, **ma)
    assert np.max(np.abs(dk_c - take(dk, cols))) <= 1e-12
    assert np.max(np.abs(dv_c - take(dv, cols))) <= 1e-12


@pytest.mark.parametrize("kind", ["causal", "padding", "sparse"])
def test_row_blocks_sum_to_full_backward(kind):
    """Row-block pieces (used to time a bounded sample) reassemble the full result."""
    B, H, N, d = 2, 1, 45, 8
    q, k, v, do = (rand((B, H, N, d), 110 + i) for i in range(4))
    ma = mask_args(kind, B, N, 115, block=16)
    o, lse = A.forward(q, k, v, 0.3, **ma)
    dq, dk, dv, _ = A.backward(q, k, v, do, 0.3, **ma)
    for b in range(B):
        dk_sum = np.zeros((N, d))
        dv_sum = np.zeros((N, d))
        for r0 in range(0, N, 10):
            r = np.arange(r0, min(N, r0 + 10))
            ob, lb, dqb, dkp, dvp = A.row_block_forward_backward(q, k, v, do, 0.3, b, 0, r, **ma)
            assert np.max(np.abs(ob - o[b, 0, r])) <= 1e-13
            fin = np.isfinite(lse[b, 0, r])
            assert np.max(np.abs((lb - lse[b, 0, r])[fin])) <= 1e-13
            assert np.max(np.abs(dqb - dq[b, 0, r])) <= 1e-12
            dk_sum += dkp
            dv_sum += dvp
        assert np.max(np.abs(dk_sum - dk[b, 0])) <= 1e-12
        assert np.max(np.abs(dv_sum - dv[b, 0])) <= 1e-12


# ---------------------------------------------------------------------------
# 15. mask orientation and boundaries, pinned without the oracle's own
#     visibility function: the expected visibility is written out by hand and
#     the attention and its derivative are computed with scalar loops.
# ---------------------------------------------------------------------------

def _brute_backward(q, k, v, do, s, vis):
    """dQ, dK, dV of L = sum(O o dO) with scalar loops over an explicit
    visibility table (the textbook derivative of the definition)."""
    n, d = len(q), len(q[0])
    p = [[0.0] * n for _ in range(n)]
    for i in range(n):
        idx = [j for j in range(n) if vis[i][j]]
        if not idx:
            continue
        logit = {j: s * sum(q[i][c] * k[j][c] for c in range(d)) for j in idx}
        mx = max(logit.values())
        tot = sum(math.exp(x - mx) for x in logit.values())
        for j in idx:
            p[i][j] = math.exp(logit[j] - mx) / tot
    dp = [[sum(do[i][c] * v[j][c] for c in range(d)) for j in range(n)] for i in range(n)]
    drow = [sum(p[i][j] * dp[i][j] for j in range(n)) for i in range(n)]
    ds = [[p[i][j] * (dp[i][j] - drow[i]) for j in range(n)] for i in range(n)]
    dq = [[s * sum(ds[i][j] * k[j][c] for j in range(n)) for c in range(d)] for i in range(n)]
    dk = [[s * sum(ds[i][j] * q[i][c] for i in range(n)) for c in range(d)] for j in range(n)]
    dv = [[sum(p[i][j] * do[i][c] for i in range(n)) for c in range(d)] for j in range(n)]
    return np.array(dq), np.array(dk), np.array(dv)


# An asymmetric tile mask (query tile i, key tile j): query tile 0 sees key
# tile 0; query tile 1 sees key tiles 0 and 1; query tile 2 sees key tiles 1
# and 2.  Its transpose differs in four places.
_TILE_MASK = np.array([[1, 0, 0],
                       [1, 1, 0],
                       [0, 1, 1]], np.uint8)
_TILE = 4
_TILE_VIS = [  # 12 x 12 by hand: row i lists the keys query i sees
    [1] * 4 + [0] * 8,
] * 4 + [
    [1] * 8 + [0] * 4,
] * 4 + [
    [0] * 4 + [1] * 8,
] * 4


def _tile_mask_error(A_):
    """Largest error of the oracle module A_ against the hand-written
    visibility: O, lse and the three gradients, block-sparse with the
    asymmetric tile mask."""
    N, d, s = 12, 3, 0.8
    q, k, v, do = (rand((1, 1, N, d), 140 + i) for i in range(4))
    o, lse = A_.forward(q, k, v, s, block_mask=_TILE_MASK, block=_TILE)
    dq, dk, dv, _ = A_.backward(q, k, v, do, s, block_mask=_TILE_MASK, block=_TILE)
    L = lambda x: x[0, 0].tolist()
    ob, lb = _brute(L(q), L(k), L(v), s, _TILE_VIS)
    gb = _brute_backward(L(q), L(k), L(v), L(do), s, _TILE_VIS)
    errs = [np.max(np.abs(o[0, 0] - ob)), np.max(np.abs(lse[0, 0] - lb))]
    errs += [np.max(np.abs(g[0, 0] - r)) for g, r in zip((dq, dk, dv), gb)]
    return max(errs)


def test_block_mask_orientation_against_hand_written_visibility():
    """The tile mask is indexed by (query tile, key tile), as the summary
    page's block-sparse extension states it ("Extension: block-sparse
    FlashAttention"): checked against a visibility table typed out by hand,
    through loops that never call the oracle's mask code."""
    assert _tile_mask_error(A) <= 1e-12
    # key tile 2 is seen by query tile 2 only: dK, dV of keys 8..11 come from
    # rows 8..11 alone; key tile 0 from rows 0..7
    N, d = 12, 3
    q, k, v, do = (rand((1, 1, N, d), 140 + i) for i in range(4))
    _, dk, dv, _ = A.backward(q, k, v, do, 0.8, block_mask=_TILE_MASK, block=_TILE)
    do_cut = do.copy()
    do_cut[0, 0, :8] = 0.0   # rows 0..7 stop contributing
    _, dk2, dv2, _ = A.backward(q, k, v, do_cut, 0.8, block_mask=_TILE_MASK, block=_TILE)
    assert np.array_equal(dv[0, 0, 8:], dv2[0, 0, 8:])
    assert np.array_equal(dk[0, 0, 8:], dk2[0, 0, 8:])
    assert np.all(dv2[0, 0, :4] == 0.0)


def _planted(monkeypatch, mistake):
    """A copy of the oracle's visibility function with one mistake planted in
    it, installed for the rest of the test."""
    real = A.visible

    def wrong(rows, n_keys, causal=False, kv_len_b=None, block_mask=None, block=128, keys=None):
        if mistake == "transposed_tile_mask" and block_mask is not None:
            block_mask = np.asarray(block_mask).T
        if mistake == "padding_off_by_one" and kv_len_b is not None:
            kv_len_b = int(kv_len_b) + 1
        return real(rows, n_keys, causal, kv_len_b, block_mask, block, keys)

    monkeypatch.setattr(A, "visible", wrong)


def test_tile_mask_pin_catches_a_transposed_mask(monkeypatch):
    _planted(monkeypatch, "transposed_tile_mask")
    assert _tile_mask_error(A) > 1e-2


def _padding_error(A_):
    """Key padding at its boundary: with kv_len = 5, key 4 is the last visible
    key and key 5 the first hidden one.  Checked against a table typed out
    by hand (j < 5) with scalar loops."""
    N, d, s, L_b = 9, 3, 0.7, 5
    q, k, v, do = (rand((1, 1, N, d), 150 + i) for i in range(4))
    o, lse = A_.forward(q, k, v, s, kv_len=np.array([L_b]))
    dq, dk, dv, _ = A_.backward(q, k, v, do, s, kv_len=np.array([L_b]))
    vis = [[1] * 5 + [0] * 4 for _ in range(N)]
    L = lambda x: x[0, 0].tolist()
    ob, lb = _brute(L(q), L(k), L(v), s, vis)
    gb = _brute_backward(L(q), L(k), L(v), L(do), s, vis)
    errs = [np.max(np.abs(o[0, 0] - ob)), np.max(np.abs(lse[0, 0] - lb))]
    errs += [np.max(np.abs(g[0, 0] - r)) for g, r in zip((dq, dk, dv), gb)]
    return max(errs), dk, dv


def test_key_padding_boundary_against_hand_written_visibility():
    err, dk, dv = _padding_error(A)
    assert err <= 1e-12
    assert np.all(dv[0, 0, 4] != 0.0) and np.all(dk[0, 0, 4] != 0.0)   # key kv_len - 1: visible
    assert np.all(dv[0, 0, 5:] == 0.0) and np.all(dk[0, 0, 5:] == 0.0)  # key kv_len: hidden


def test_padding_pin_catches_an_off_by_one(monkeypatch):
    _planted(monkeypatch, "padding_off_by_one")
    assert _padding_error(A)[0] > 1e-2
