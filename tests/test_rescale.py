"""GPU parity on inputs whose running row maximum grows past the lazy-rescale
threshold at every key tile.

The forward kernels keep O unnormalised and rescale it only when a row's
maximum grows by more than 8 in log2 units (so that P~ = 2^(c S - m) stays
below 2^8).  On random inputs that happens almost only at the first key tile.
Here the scores climb by about 9 log2 units from one 128-key tile to the next,
with a spread of 4 inside each tile, so every tile of every row rescales O
(both 64-key halves of a tile, at d = 64 and d = 128).  At d = 128 the
rescale must wait for the previous tile's P~ V: the next score tile may have
been computed before it.  An O rescaled too early keeps the previous tile's
P~ V unscaled, about 2^9 times too heavy, which the oracle comparison cannot
miss.

The backward runs on the same inputs.  O, lse, dK and dV are held to the usual
tolerances.  dQ is not, and for a reason these inputs make plain: a row's
visible keys share a large common component along the score direction, and
dQ_i = c sum_j dS_ij k_j with sum_j dS_ij = 0, so dQ is the small remainder of
large terms.  Two roundings that the kernels make by design do not cancel
there: dS goes to the tensor core in bf16 (relative rounding at most 2^-9 per
element), and D = rowsum(dO o O) is taken from O as stored in bf16, so that
every dS of row i carries -P_ij dD_i.  dQ is therefore held, element by
element, to the bound those two roundings give (each with a factor of two, and
the fp32 error of dP - D beside them) plus its own bf16 output rounding."""
import numpy as np
import pytest

import oracle
from workloads import bf16_round
from _gpu_helpers import TOL, f64, max_abs, rel_fro, run, to_device


def growing_case(B, H, N, d, seed, step_log2=9.0, spread_log2=4.0, kv_len=None):
    """q has a constant component a on its first coordinate; key j's first
    coordinate is (step * (j // 128) + spread * u_j) / (c a), u_j uniform in
    [0, 1), c = d^-1/2 log2 e: the score of every query row with key j is then
    that many log2 units plus a small random part."""
    rng = np.random.default_rng(seed)
    c = d ** -0.5 * np.log2(np.e)
    a = 4.0
    x = {n: rng.standard_normal((B, H, N, d)).astype(np.float32) * np.float32(0.1)
         for n in ("q", "k")}
    x["q"][..., 0] = a
    tile = np.arange(N) // 128
    x["k"][..., 0] = (step_log2 * tile + spread_log2 * rng.random((B, H, N))) / (c * a)
    for n in ("v", "do"):
        x[n] = rng.standard_normal((B, H, N, d)).astype(np.float32)
    out = {}
    for n in ("q", "k", "v", "do"):
        out[n], out[n + "_bits"] = bf16_round(x[n])
    out["kv_len"] = None if kv_len is None else np.asarray(kv_len, np.int32)
    out["block_mask"] = None
    return out


def test_scores_climb_past_the_threshold_at_every_tile():
    """The construction does what the docstring says (checked on the host): the
    largest log2-unit score of each 128-key tile exceeds the previous tile's by
    more than 8 for every query row."""
    B, H, N, d = 1, 1, 1024, 128
    case = growing_case(B, H, N, d, seed=1)
    c = d ** -0.5 * np.log2(np.e)
    s = c * np.einsum("qd,kd->qk", case["q"][0, 0], case["k"][0, 0])
    tmax = s.reshape(N, N // 128, 128).max(axis=2)
    assert np.all(np.diff(tmax, axis=1) > 8.0)


CASES = [  # d, causal, kv_len
    (128, False, None),
    (128, True, None),
    (64, False, None),
    (64, True, None),
    (128, False, [900]),
]


def dq_rounding_bound(case, scale, causal, dq_ref, D_ref, o_ref):
    """Per element of dQ: c (2^-8 |dS| + 1e-6 P (|dP| + |D|)) |K|
    + c dD (P |K|) + 2^-8 |dQ| + 1e-5, with dD_i = 2^-8 sum_c |dO_ic O_ic|, from
    the oracle's O, P, dP, D and dS of each (batch, head)."""
    q, k, v, do = (np.asarray(case[n], np.float64) for n in ("q", "k", "v", "do"))
    B, H, N, _ = q.shape
    bound = np.empty_like(dq_ref)
    for b in range(B):
        kv_b = None if case["kv_len"] is None else int(case["kv_len"][b])
        vis = oracle.visible(N, N, causal=causal, kv_len_b=kv_b)
        for h in range(H):
            p, _ = oracle.probabilities(oracle.scores(q[b, h], k[b, h], scale, vis))
            dp = do[b, h] @ v[b, h].T
            dd = D_ref[b, h][:, None]
            ds = p * (dp - dd)
            err_ds = 2.0 ** -8 * np.abs(ds) + 1e-6 * p * (np.abs(dp) + np.abs(dd))
            err_d = 2.0 ** -8 * np.sum(np.abs(do[b, h] * o_ref[b, h]), axis=1)[:, None]
            ak = np.abs(k[b, h])
            bound[b, h] = (scale * (err_ds @ ak) + scale * err_d * (p @ ak)
                           + 2.0 ** -8 * np.abs(dq_ref[b, h]) + 1e-5)
    return bound


@pytest.mark.gpu
@pytest.mark.parametrize("d,causal,kv_len", CASES)
def test_rescale_at_every_tile(fa, d, causal, kv_len):
    B, H, N = 1, 2, 1024
    scale = d ** -0.5
    case = growing_case(B, H, N, d, seed=40 + d + causal, kv_len=kv_len)
    t = to_device(case, "bf16")
    o, lse, (dq, dk, dv) = run(fa, t, scale, causal)
    kw = dict(causal=causal, kv_len=case["kv_len"])
    ro, rl = oracle.forward(case["q"], case["k"], case["v"], scale, **kw)
    to, tl, tg = TOL["bf16"]
    assert max_abs(f64(o), ro) <= to, ("O", max_abs(f64(o), ro))
    e_l = max_abs(lse.cpu().numpy().astype(np.float64), rl, finite_only=True)
    assert e_l <= tl, ("lse", e_l)
    rdq, rdk, rdv, rD = oracle.backward(case["q"], case["k"], case["v"], case["do"], scale, **kw)
    for name, g, r in (("dK", dk, rdk), ("dV", dv, rdv)):
        assert rel_fro(f64(g), r) <= tg, (name, rel_fro(f64(g), r))
    err = np.abs(f64(dq) - rdq)
    bound = dq_rounding_bound(case, scale, causal, rdq, rD, ro)
    assert np.all(err <= bound), ("dQ", float((err / bound).max()))
