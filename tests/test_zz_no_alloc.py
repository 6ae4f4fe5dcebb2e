"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (for example a plugin whose host framework has reserved all device
memory for its own pool, or latency-critical code that must not call
cudaMalloc because it can synchronize the device).  It works in a fixed
scratch array inside the library instead of a caller-provided workspace.

Checked through the C ABI against fa_bwd with an allocated workspace, on
calls in a row with different inputs, sizes, masks and streams (the scratch
keeps the previous call's contents, so no call may depend on them).  The
backward is deterministic -- every dQ, dK, dV row is summed by one CTA in a
fixed order -- so the two entry points must agree bit for bit; one call is
also compared with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from workloads import random_case
from _gpu_helpers import TOL, f64, rel_fro, to_device

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.view(torch.int16)


def _both(fa, case, B, H, N, d, causal, stream=None):
    """fa.backward (fa_bwd, allocated workspace) and fa_bwd_noalloc on the same
    inputs; the second on `stream` when one is given."""
    t = to_device(case, "bf16")
    scale = d ** -0.5
    mk = dict(kv_len=t["kv_len"], block_mask=t["block_mask"])
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, causal, **mk)
    ref = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal, **mk)
    torch.cuda.synchronize()
    got = [torch.full_like(t["q"], float("nan")) for _ in range(3)]
    mask = fa.make_mask(**mk)
    s = stream if stream is not None else torch.cuda.current_stream()
    with torch.cuda.stream(s):
        fa.fa_bwd_noalloc(t["q"], t["k"], t["v"], o, t["do"], lse, got[0], got[1], got[2],
                          B, H, N, d, scale, causal, mask, stream=s)
    s.synchronize()
    code, site = fa.fa_get_device_status()
    assert code == 0, (code, site)
    return ref, got


def test_noalloc_backward_matches_fa_bwd_twice(fa):
    # first call: 2 x 4 heads of 1000 tokens, causal (32 KB of scratch)
    case = random_case(2, 4, 1000, 64, seed=31)
    ref, got = _both(fa, case, 2, 4, 1000, 64, True)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(_bits(g), _bits(r)), name
    # the same call against the oracle, within the bf16 tolerance
    rdq, rdk, rdv, _ = oracle.backward(case["q"], case["k"], case["v"], case["do"], 64 ** -0.5,
                                       causal=True)
    for name, g, r in zip(("dQ", "dK", "dV"), got, (rdq, rdk, rdv)):
        assert rel_fro(f64(g), r) <= TOL["bf16"][2], name
    # second call right after: other inputs, other size, non-causal
    ref, got = _both(fa, random_case(1, 3, 777, 128, seed=32), 1, 3, 777, 128, False)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.all(np.isfinite(f64(g))), name
        assert torch.equal(_bits(g), _bits(r)), name


def test_noalloc_with_masks_and_a_side_stream(fa):
    # key padding: the scratch holds D of padded query rows too
    kv = np.array([700, 130, 1], np.int32)
    case = random_case(3, 2, 700, 64, seed=33, kv_len=kv)
    ref, got = _both(fa, case, 3, 2, 700, 64, False)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(_bits(g), _bits(r)), name
    # block-sparse (rows with no visible tile), on a non-default stream
    bm = np.array([[0, 0, 0, 0], [1, 1, 0, 0], [0, 1, 1, 1], [1, 0, 0, 1]], np.uint8)
    case = random_case(1, 3, 500, 128, seed=34, block_mask=bm)
    side = torch.cuda.Stream()
    ref, got = _both(fa, case, 1, 3, 500, 128, False, stream=side)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(_bits(g), _bits(r)), name


def test_noalloc_rejects_sizes_beyond_its_scratch(fa):
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(16, dtype=torch.float32, device="cuda")
    B, H, N, d = 64, 16, 16384, 128   # D alone needs 64 MiB: more than the fixed scratch
    assert fa.fa_bwd_workspace_size(B, H, N, d) > fa.NOALLOC_SCRATCH_BYTES
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd_noalloc(x, x, x, x, x, lse, x, x, x, B, H, N, d, 0.1, True)
    assert e.value.code == 2   # FA_ERR_UNSUPPORTED, rejected before any launch
