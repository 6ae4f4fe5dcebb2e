"""Block-sparse work order (fa_block_mask_order and fa_mask.tile_order).

The order is integer work: it is checked bit for bit against a stable sort of
the tile counts written here with numpy.  Taking the tiles in any order must
leave every output bit-identical, since each tile's result does not depend on
which CTA computes it; that is checked for the computed order, for random
permutations, with and without the causal restriction, at d = 64 and 128."""
import numpy as np
import pytest
import torch

from workloads import block_mask_pattern, random_case
from _gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def expected_order(bm, causal):
    """Query tiles, then key tiles, most visible tiles first, ties by index (a
    stable sort of the negated counts)."""
    T = bm.shape[0]
    vis = bm != 0
    if causal:
        vis = vis & (np.arange(T)[None, :] <= np.arange(T)[:, None])
    rows = vis.sum(axis=1)
    cols = vis.sum(axis=0)
    order = lambda c: np.argsort(-c, kind="stable")
    return np.concatenate([order(rows), order(cols)]).astype(np.int32)


MASKS = [("random", 1), ("random", 5), ("random", 128), ("random", 130), ("local_global", 128),
         ("butterfly", 64), ("strided", 37), ("local", 512),
         ("random", 4096), ("local_global", 4095)]  # the largest side: 64 KB of shared memory


@pytest.mark.parametrize("pattern,T", MASKS)
@pytest.mark.parametrize("causal", [False, True])
def test_order_is_the_stable_sort_of_the_counts(fa, pattern, T, causal):
    rng = np.random.default_rng(T * 7 + causal)
    bm = block_mask_pattern(pattern, T, rng)
    out = fa.block_mask_order(torch.from_numpy(bm).cuda(), causal)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert got.shape == (fa.fa_block_mask_order_len(T),)
    assert np.array_equal(got, expected_order(bm, causal))


def _run(fa, t, scale, causal, order):
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, causal, block_mask=t["block_mask"],
                        tile_order=order)
    g = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal,
                    block_mask=t["block_mask"], tile_order=order)
    torch.cuda.synchronize()
    code, site = fa.fa_get_device_status()
    assert code == 0, "device status %d at site %d" % (code, site)
    return (o, lse) + tuple(g)


@pytest.mark.parametrize("d,causal,pattern", [(64, False, "local_global"), (64, True, "random"),
                                              (128, False, "local_global"),
                                              (128, True, "butterfly")])
def test_outputs_do_not_depend_on_the_order(fa, d, causal, pattern):
    B, H, N = 2, 3, 2048 - 37  # ragged last tile; T = 16
    T = (N + 127) // 128
    bm = block_mask_pattern(pattern, T, np.random.default_rng(d + causal), p=0.3)
    case = random_case(B, H, N, d, seed=11 * d + causal, block_mask=bm)
    t = to_device(case, "bf16")
    scale = d ** -0.5
    ref = _run(fa, t, scale, causal, None)
    computed = fa.block_mask_order(t["block_mask"], causal)
    rng = np.random.default_rng(5)
    perm = np.concatenate([rng.permutation(T), rng.permutation(T)]).astype(np.int32)
    for order in (computed, torch.from_numpy(perm).cuda()):
        got = _run(fa, t, scale, causal, order)
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), got, ref):
            assert torch.equal(a, b), name


def test_order_with_dropout_and_fp32_paths(fa):
    """The kernels with dropout read the order too; the fp32 path ignores it."""
    B, H, N, d = 1, 2, 1024, 64
    T = N // 128
    bm = block_mask_pattern("local_global", T)
    for dtype, drop in (("bf16", 0.2), ("fp32", 0.0)):
        case = random_case(B, H, N, d, seed=3, dtype=dtype, block_mask=bm)
        t = to_device(case, dtype)
        order = fa.block_mask_order(t["block_mask"], False)
        outs = []
        for tile_order in (None, order):
            o, lse = fa.forward(t["q"], t["k"], t["v"], 0.125, False, block_mask=t["block_mask"],
                                dropout_p=drop, seed=9, offset=1, tile_order=tile_order)
            g = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, 0.125, False,
                            block_mask=t["block_mask"], dropout_p=drop, seed=9, offset=1,
                            tile_order=tile_order)
            torch.cuda.synchronize()
            outs.append((o, lse) + tuple(g))
        for a, b in zip(*outs):
            assert torch.equal(a, b)
